// C ABI: descriptor validation, kernel choice, workspace layout, dispatch.
//
// Validation follows the fault-tolerance rules of
// githubissues.com/ysh329/OpenCL-101/52 ("init fault tolerance" and the
// uninitialised-activation bug case): every field is checked, unknown enum
// values are rejected, and nothing is launched for a rejected call.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <initializer_list>

#include "internal.h"

namespace gbconv {

bool log_enabled() {
    static const bool on = [] {
        const char *v = std::getenv("GBCONV_LOG");
        return v && v[0] && std::strcmp(v, "0") != 0;
    }();
    return on;
}

void log_line(const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    std::fprintf(stderr, "gbconv: %s\n", buf);
}

namespace {

int64_t out_extent(int64_t in, int k, int pad, int stride) {
    int64_t span = in + 2 * (int64_t)pad - k;
    if (span < 0) return 0;
    return span / stride + 1;
}

bool in_range(int v, int lo, int hi) { return v >= lo && v <= hi; }

// a * b when it is at most `limit` (a, b >= 0), else -1: element counts are
// formed without signed overflow, so a huge shape cannot wrap past the limit.
int64_t mul_capped(int64_t a, int64_t b, int64_t limit) {
    if (a < 0 || b < 0) return -1;
    if (b != 0 && a > limit / b) return -1;
    return a * b;
}
int64_t elems_capped(std::initializer_list<int64_t> factors, int64_t limit) {
    int64_t n = 1;
    for (int64_t f : factors) {
        n = mul_capped(n, f, limit);
        if (n < 0) return -1;
    }
    return n;
}

// The tensor-core path for this problem, within CUDA's grid limits: the
// element-wise split of channels-last fp32 x runs one 256-thread CTA per 256
// elements of its [N][S][Cs] half, in a 1-D grid.
bool tc_ok(const Problem &q) {
    if (!tc_supported(q)) return false;
    if (q.dtype == GBCONV_F32 && q.cl) {
        const int64_t n = (int64_t)q.N * q.in_vol * tc_split_half(q.C);
        if ((n + 255) / 256 > 0x7FFFFFFF) return false;
    }
    return true;
}

// Structural validation: shapes and enums only (no pointers).
gbconv_status build_problem(const gbconv_desc *d, int ndim, Problem *p) {
    if (!d) return GBCONV_ERR_NULL;
    if (ndim != 2 && ndim != 3) return GBCONV_ERR_SHAPE;
    if ((d->flags & ~(GBCONV_FLAG_TPAD_MASK | GBCONV_FLAG_MAXPOOL2 | GBCONV_FLAG_CHANNELS_LAST)) != 0)
        return GBCONV_ERR_RESERVED;
    const int cl = (d->flags & GBCONV_FLAG_CHANNELS_LAST) ? 1 : 0;
    const int pool = (d->flags & GBCONV_FLAG_MAXPOOL2) ? 1 : 0;
    if (pool && ndim != 2) return GBCONV_ERR_SHAPE;
    const int tpad = d->flags & GBCONV_FLAG_TPAD_MASK;
    if (tpad > GBCONV_TPAD_NONE) return GBCONV_ERR_RESERVED;
    if (ndim == 2 && tpad != GBCONV_TPAD_SYMMETRIC) return GBCONV_ERR_SHAPE;
    if (!in_range(d->dtype, GBCONV_F32, GBCONV_BF16)) return GBCONV_ERR_DTYPE;
    if (!in_range(d->act, GBCONV_ACT_NONE, GBCONV_ACT_RELU)) return GBCONV_ERR_ACT;
    if (!in_range(d->w_layout, GBCONV_W_OIHW, GBCONV_W_PACKED)) return GBCONV_ERR_LAYOUT;
    if (!in_range(d->algo, GBCONV_ALGO_AUTO, GBCONV_ALGO_DIRECT_TC)) return GBCONV_ERR_ALGO;
    const int dims[] = {d->N, d->C, d->D, d->H, d->W, d->OC};
    for (int v : dims)
        if (!in_range(v, 1, GBCONV_MAX_DIM)) return GBCONV_ERR_SHAPE;
    if (ndim == 2 && d->D != 1) return GBCONV_ERR_SHAPE;
    if (!in_range(d->k, 1, GBCONV_MAX_K)) return GBCONV_ERR_SHAPE;
    if (!in_range(d->stride, 1, GBCONV_MAX_STRIDE)) return GBCONV_ERR_SHAPE;
    if (!in_range(d->pad, 0, GBCONV_MAX_K)) return GBCONV_ERR_SHAPE;

    Problem q{};
    q.ndim = ndim;
    q.N = d->N; q.C = d->C; q.D = d->D; q.H = d->H; q.W = d->W;
    q.OC = d->OC; q.k = d->k; q.pad = d->pad; q.stride = d->stride;
    q.kd = ndim == 3 ? d->k : 1;
    q.pad_d = q.pad_d_back = 0;
    if (ndim == 3) {
        q.pad_d = tpad == GBCONV_TPAD_SYMMETRIC ? d->pad : (tpad == GBCONV_TPAD_CAUSAL ? d->k - 1 : 0);
        q.pad_d_back = tpad == GBCONV_TPAD_SYMMETRIC ? d->pad : 0;
    }
    int64_t od = 1;
    if (ndim == 3) {
        const int64_t span = (int64_t)d->D + q.pad_d + q.pad_d_back - d->k;
        od = span < 0 ? 0 : span / d->stride + 1;
    }
    int64_t oh = out_extent(d->H, d->k, d->pad, d->stride);
    int64_t ow = out_extent(d->W, d->k, d->pad, d->stride);
    if (od <= 0 || oh <= 0 || ow <= 0) return GBCONV_ERR_SHAPE;
    q.OD = (int)od; q.OH = (int)oh; q.OW = (int)ow;
    q.taps = q.kd * q.k * q.k;
    q.in_vol = (int64_t)q.D * q.H * q.W;
    q.out_vol = od * oh * ow;
    q.pool = pool;
    q.cl = cl;
    q.YH = pool ? q.OH / 2 : q.OH;
    q.YW = pool ? q.OW / 2 : q.OW;
    if (q.YH <= 0 || q.YW <= 0) return GBCONV_ERR_SHAPE;
    q.x_elems = elems_capped({q.N, q.C, q.D, q.H, q.W}, GBCONV_MAX_ELEMS);
    q.w_elems = elems_capped({q.OC, q.C, q.taps}, GBCONV_MAX_ELEMS);
    q.y_elems = elems_capped({q.N, q.OC, q.OD, q.YH, q.YW}, GBCONV_MAX_ELEMS);
    if (q.x_elems < 0 || q.w_elems < 0 || q.y_elems < 0) return GBCONV_ERR_SHAPE;
    q.dtype = d->dtype; q.act = d->act; q.w_layout = d->w_layout;
    q.elt = d->dtype == GBCONV_F32 ? 4 : 2;

    // Kernel choice. Small reduction depth (IC * kvol) is bandwidth-bound
    // work: the direct kernel. Otherwise an implicit GEMM: tensor cores for
    // 16-bit storage; for fp32 the tensor cores' three TF32 products while
    // the reduction is at most kTf32x3AutoMaxK products long, exact fp32 FMA
    // on the CUDA cores beyond. (The three-product error grows with the
    // reduction: measured relative L2 error at most 7.2e-6 up to 1,000
    // products and up to 1.6e-5 beyond, against 1e-5 for fp32; the CUDA-core
    // GEMM stays below 1e-6.)
    constexpr int64_t kTf32x3AutoMaxK = 1000;
    const bool tf32x3_ok = q.dtype != GBCONV_F32 || (int64_t)q.C * q.taps <= kTf32x3AutoMaxK;
    int algo = d->algo;
    if (algo == GBCONV_ALGO_AUTO && q.cl) {
        // Channels-last: the implicit GEMMs only (the direct kernels read NCHW).
        algo = ((q.dtype == GBCONV_F32 || tc_cl_direct(q)) && tc_ok(q) && tf32x3_ok) ? GBCONV_ALGO_IGEMM_TC
                                                                                    : GBCONV_ALGO_IGEMM_FFMA;
    } else if (algo == GBCONV_ALGO_AUTO) {
        // fp32 3x3 stems of 16+ output channels: the tensor-core stem
        // (measured faster than the CUDA-core stem from 16 to 128 channels
        // on 640 x 640 images, stride 1 and 2).
        if (q.pool)
            algo = GBCONV_ALGO_DIRECT;          // the fused pool's only kernel
        else if (stem_tc_supported(q) && q.OC >= 16)
            algo = GBCONV_ALGO_DIRECT_TC;
        else if ((int64_t)q.C * q.taps <= 64 && direct_supported(q))
            algo = GBCONV_ALGO_DIRECT;
        else if (tc_ok(q) && tf32x3_ok)
            algo = GBCONV_ALGO_IGEMM_TC;       // fp32: three TF32 products
        else
            algo = GBCONV_ALGO_IGEMM_FFMA;
    }
    q.algo = algo;
    if (algo == GBCONV_ALGO_DIRECT && !direct_supported(q)) return GBCONV_ERR_ALGO;
    if (algo == GBCONV_ALGO_IGEMM_TC && !tc_ok(q)) return GBCONV_ERR_ALGO;
    if (algo == GBCONV_ALGO_DIRECT_TC && !stem_tc_supported(q)) return GBCONV_ERR_ALGO;
    if (q.cl && !(algo == GBCONV_ALGO_IGEMM_FFMA ||
                  (algo == GBCONV_ALGO_IGEMM_TC && (tc_cl_direct(q) || q.dtype == GBCONV_F32))))
        return GBCONV_ERR_ALGO;
    // The fused pool lives in the few-channel 3x3 direct kernel only.
    if (q.pool && !(algo == GBCONV_ALGO_DIRECT && stem_supported(q))) return GBCONV_ERR_ALGO;
    *p = q;
    return GBCONV_OK;
}

bool aligned(const void *ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

bool overlap(const void *a, size_t an, const void *b, size_t bn) {
    if (!a || !b || an == 0 || bn == 0) return false;
    uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + bn && b0 < a0 + an;
}

gbconv_status device_check() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GBCONV_ERR_UNSUPPORTED_DEVICE;
    }
    return gbconv_device_supported(dev) ? GBCONV_OK : GBCONV_ERR_UNSUPPORTED_DEVICE;
}

gbconv_status forward(const gbconv_desc *d, int ndim, const void *x,
                      const void *w, const float *b, void *y, cudaStream_t s) {
    Problem p;
    gbconv_status st = build_problem(d, ndim, &p);
    if (st != GBCONV_OK) return st;
    if (!x || !w || !y) return GBCONV_ERR_NULL;
    if (!aligned(x, p.elt) || !aligned(w, p.elt) || !aligned(y, p.elt) ||
        (b && !aligned(b, 4)))
        return GBCONV_ERR_ALIGN;
    if (p.w_layout == GBCONV_W_PACKED && !aligned(w, 256)) return GBCONV_ERR_ALIGN;
    // The tensor-core kernel reads channels-last x in place with TMA.
    if (p.algo == GBCONV_ALGO_IGEMM_TC && tc_cl_direct(p) && !aligned(x, 16)) return GBCONV_ERR_ALIGN;
    const size_t xb = (size_t)p.x_elems * p.elt, yb = (size_t)p.y_elems * p.elt;
    const size_t wb = p.w_layout == GBCONV_W_PACKED ? packed_weight_bytes(p)
                                                    : (size_t)p.w_elems * p.elt;
    Workspace ws = workspace_layout(p);
    if (ws.total > 0) {
        if (!d->workspace || d->workspace_bytes < ws.total) return GBCONV_ERR_WORKSPACE;
        if (!aligned(d->workspace, 256)) return GBCONV_ERR_WORKSPACE;
    }
    // The kernels write y and the workspace while they read x, w and b.
    const size_t bb = b ? (size_t)p.OC * 4 : 0;
    if (overlap(y, yb, x, xb) || overlap(y, yb, w, wb) || overlap(y, yb, b, bb) ||
        overlap(y, yb, d->workspace, ws.total) || overlap(d->workspace, ws.total, x, xb) ||
        overlap(d->workspace, ws.total, w, wb) || overlap(d->workspace, ws.total, b, bb))
        return GBCONV_ERR_OVERLAP;
    if (log_enabled())
        log_line("conv%dd N=%d C=%d D=%d H=%d W=%d OC=%d k=%d pad=%d stride=%d dtype=%d act=%d%s%s%s "
                 "-> OD=%d OH=%d OW=%d algo=%s weights=%s workspace=%zu",
                 ndim, p.N, p.C, p.D, p.H, p.W, p.OC, p.k, p.pad, p.stride, p.dtype, p.act,
                 p.cl ? " channels_last" : "", p.pool ? " maxpool2" : "",
                 p.pad_d != p.pad && ndim == 3 ? " frame_pad" : "", p.OD, p.YH, p.YW,
                 gbconv_algo_name(p.algo), p.w_layout == GBCONV_W_PACKED ? "packed" : "oihw", ws.total);
    st = device_check();
    if (st != GBCONV_OK) return st;

    char *wsp = static_cast<char *>(d->workspace);
    cudaError_t e = cudaSuccess;
    switch (p.algo) {
    case GBCONV_ALGO_DIRECT:
        // The direct kernel reads OIHW; its packed form is an OIHW copy.
        e = launch_direct(p, x, w, b, y, s);
        break;
    case GBCONV_ALGO_DIRECT_TC:
        // Reads OIHW as well (the tensor-core tiles are built in the kernel).
        e = launch_stem_tc(p, x, w, b, y, s);
        break;
    case GBCONV_ALGO_IGEMM_FFMA: {
        const void *wp = w;
        if (p.w_layout == GBCONV_W_OIHW) {
            e = launch_pack_ffma(p, w, wsp + ws.w_off, s);
            wp = wsp + ws.w_off;
        }
        float *part = ws.part_bytes ? reinterpret_cast<float *>(wsp + ws.part_off) : nullptr;
        if (e == cudaSuccess) e = launch_igemm_ffma(p, x, wp, b, y, part, ffma_split_slices(p), s);
        break;
    }
    case GBCONV_ALGO_IGEMM_TC: {
        const bool oihw = p.w_layout == GBCONV_W_OIHW;
        const void *wp = oihw ? static_cast<const void *>(wsp + ws.w_off) : w;
        if (tc_cl_direct(p)) {
            if (oihw) e = launch_pack_tc(p, w, wsp + ws.w_off, s);
            if (e == cudaSuccess) e = launch_igemm_tc(p, x, wp, b, y, s);
        } else {
            // the weight pack and the x layout pass share one launch
            e = oihw ? launch_prep_tc(p, w, wsp + ws.w_off, x, wsp + ws.x_off, s)
                     : launch_to_channels_last(p, x, wsp + ws.x_off, s);
            if (e == cudaSuccess) e = launch_igemm_tc(p, wsp + ws.x_off, wp, b, y, s);
        }
        break;
    }
    default:
        return GBCONV_ERR_ALGO;
    }
    return launch_status(e);
}

}  // namespace

gbconv_status make_problem(const gbconv_desc *d, int ndim, Problem *p) {
    return build_problem(d, ndim, p);
}

size_t packed_weight_bytes(const Problem &p) {
    switch (p.algo) {
    case GBCONV_ALGO_DIRECT:
    case GBCONV_ALGO_DIRECT_TC:
        return (size_t)p.w_elems * p.elt;
    case GBCONV_ALGO_IGEMM_FFMA:
        return (size_t)p.taps * p.C * ffma_ocpad(p.OC) * p.elt;
    case GBCONV_ALGO_IGEMM_TC:
        return (size_t)p.taps * p.OC * tc_row_channels(p) * p.elt;
    }
    return 0;
}

Workspace workspace_layout(const Problem &p) {
    Workspace ws;
    size_t off = 0;
    if (p.algo == GBCONV_ALGO_IGEMM_TC && !tc_cl_direct(p)) {
        // channels-last copy of x (16-bit) or its hi/lo split (fp32)
        ws.x_off = off;
        ws.x_bytes = (size_t)p.N * p.in_vol * tc_row_channels(p) * p.elt;
        off = align256(off + ws.x_bytes);
    }
    if (p.w_layout == GBCONV_W_OIHW && p.algo != GBCONV_ALGO_DIRECT && p.algo != GBCONV_ALGO_DIRECT_TC) {
        ws.w_off = off;
        ws.w_bytes = packed_weight_bytes(p);
        off = align256(off + ws.w_bytes);
    }
    if (p.algo == GBCONV_ALGO_IGEMM_FFMA && ffma_split_slices(p) > 0) {
        ws.part_off = off;
        ws.part_bytes = (size_t)ffma_split_slices(p) * p.OC * p.N * p.out_vol * sizeof(float);
        off = align256(off + ws.part_bytes);
    }
    ws.total = off;
    return ws;
}

}  // namespace gbconv

using namespace gbconv;

extern "C" {

gbconv_status gbconv_conv2d_fwd(const gbconv_desc *desc, const void *x,
                                const void *w, const float *b, void *y,
                                cudaStream_t stream) {
    return forward(desc, 2, x, w, b, y, stream);
}

gbconv_status gbconv_conv3d_fwd(const gbconv_desc *desc, const void *x,
                                const void *w, const float *b, void *y,
                                cudaStream_t stream) {
    return forward(desc, 3, x, w, b, y, stream);
}

gbconv_status gbconv_output_shape(const gbconv_desc *desc, int ndim, int *OD,
                                  int *OH, int *OW) {
    Problem p;
    gbconv_status st = build_problem(desc, ndim, &p);
    if (st != GBCONV_OK) return st;
    if (!OD || !OH || !OW) return GBCONV_ERR_NULL;
    *OD = p.OD; *OH = p.YH; *OW = p.YW;
    return GBCONV_OK;
}

gbconv_status gbconv_workspace_size(const gbconv_desc *desc, int ndim,
                                    size_t *bytes) {
    Problem p;
    gbconv_status st = build_problem(desc, ndim, &p);
    if (st != GBCONV_OK) return st;
    if (!bytes) return GBCONV_ERR_NULL;
    *bytes = workspace_layout(p).total;
    return GBCONV_OK;
}

gbconv_status gbconv_weight_packed_size(const gbconv_desc *desc, int ndim,
                                        size_t *bytes) {
    Problem p;
    gbconv_status st = build_problem(desc, ndim, &p);
    if (st != GBCONV_OK) return st;
    if (!bytes) return GBCONV_ERR_NULL;
    *bytes = packed_weight_bytes(p);
    return GBCONV_OK;
}

gbconv_status gbconv_weight_pack(const gbconv_desc *desc, int ndim,
                                 const void *w_oihw, void *w_packed,
                                 cudaStream_t stream) {
    Problem p;
    gbconv_status st = build_problem(desc, ndim, &p);
    if (st != GBCONV_OK) return st;
    if (!w_oihw || !w_packed) return GBCONV_ERR_NULL;
    if (!aligned(w_oihw, p.elt) || !aligned(w_packed, 256)) return GBCONV_ERR_ALIGN;
    if (overlap(w_oihw, (size_t)p.w_elems * p.elt, w_packed, packed_weight_bytes(p)))
        return GBCONV_ERR_OVERLAP;
    st = device_check();
    if (st != GBCONV_OK) return st;
    cudaError_t e;
    switch (p.algo) {
    case GBCONV_ALGO_DIRECT:
    case GBCONV_ALGO_DIRECT_TC:
        e = cudaMemcpyAsync(w_packed, w_oihw, (size_t)p.w_elems * p.elt,
                            cudaMemcpyDeviceToDevice, stream);
        break;
    case GBCONV_ALGO_IGEMM_FFMA:
        e = launch_pack_ffma(p, w_oihw, w_packed, stream);
        break;
    default:
        e = launch_pack_tc(p, w_oihw, w_packed, stream);
        break;
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GBCONV_ERR_LAUNCH;
    }
    return GBCONV_OK;
}

gbconv_status gbconv_fold_batchnorm(const gbconv_desc *desc, int ndim, const void *w,
                                    const float *b, const float *gamma, const float *beta,
                                    const float *mean, const float *var, float eps,
                                    void *w_out, float *b_out, cudaStream_t stream) {
    Problem p;
    gbconv_status st = build_problem(desc, ndim, &p);
    if (st != GBCONV_OK) return st;
    if (!w || !gamma || !beta || !mean || !var || !w_out || !b_out) return GBCONV_ERR_NULL;
    if (!(eps >= 0.0f) || eps > 3.0e38f) return GBCONV_ERR_SHAPE;
    if (!aligned(w, p.elt) || !aligned(w_out, p.elt) || !aligned(b_out, 4) || !aligned(gamma, 4) ||
        !aligned(beta, 4) || !aligned(mean, 4) || !aligned(var, 4) || (b && !aligned(b, 4)))
        return GBCONV_ERR_ALIGN;
    const size_t wb = (size_t)p.w_elems * p.elt, vb = (size_t)p.OC * 4;
    // w_out may be w and b_out may be b (in place); nothing else may overlap.
    if ((w_out != w && overlap(w_out, wb, w, wb)) || (b_out != b && overlap(b_out, vb, b, b ? vb : 0)) ||
        overlap(w_out, wb, b_out, vb) || overlap(w_out, wb, gamma, vb) || overlap(w_out, wb, beta, vb) ||
        overlap(w_out, wb, mean, vb) || overlap(w_out, wb, var, vb) || overlap(b_out, vb, gamma, vb) ||
        overlap(b_out, vb, beta, vb) || overlap(b_out, vb, mean, vb) || overlap(b_out, vb, var, vb) ||
        overlap(b_out, vb, w, wb))
        return GBCONV_ERR_OVERLAP;
    st = device_check();
    if (st != GBCONV_OK) return st;
    if (launch_fold_bn(p, w, b, gamma, beta, mean, var, eps, w_out, b_out, stream) != cudaSuccess) {
        cudaGetLastError();
        return GBCONV_ERR_LAUNCH;
    }
    return GBCONV_OK;
}

gbconv_status gbconv_select_algo(const gbconv_desc *desc, int ndim, int *algo) {
    Problem p;
    gbconv_status st = build_problem(desc, ndim, &p);
    if (st != GBCONV_OK) return st;
    if (!algo) return GBCONV_ERR_NULL;
    *algo = p.algo;
    return GBCONV_OK;
}

int gbconv_device_supported(int device) {
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (device < 0 || device >= n) return 0;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return (major == 10 && minor == 3) ? 1 : 0;
}

const char *gbconv_status_string(gbconv_status s) {
    switch (s) {
    case GBCONV_OK: return "ok";
    case GBCONV_ERR_NULL: return "null pointer";
    case GBCONV_ERR_SHAPE: return "invalid shape";
    case GBCONV_ERR_DTYPE: return "invalid dtype";
    case GBCONV_ERR_ACT: return "invalid activation";
    case GBCONV_ERR_ALIGN: return "misaligned pointer";
    case GBCONV_ERR_WORKSPACE: return "workspace missing, short or misaligned";
    case GBCONV_ERR_UNSUPPORTED_DEVICE: return "unsupported device (need compute capability 10.3)";
    case GBCONV_ERR_LAUNCH: return "kernel launch failed";
    case GBCONV_ERR_TIMEOUT: return "device-side wait timed out";
    case GBCONV_ERR_ALGO: return "algorithm unknown or not applicable";
    case GBCONV_ERR_LAYOUT: return "invalid weight layout";
    case GBCONV_ERR_OVERLAP: return "output overlaps an input or the workspace";
    case GBCONV_ERR_CUDA: return "CUDA call failed";
    case GBCONV_ERR_RESERVED: return "reserved flag bit set or unknown frame-padding mode";
    case GBCONV_ERR_TOO_LARGE: return "problem needs more scratch than the fixed no-allocation array holds";
    }
    return "unknown status";
}

const char *gbconv_algo_name(int algo) {
    switch (algo) {
    case GBCONV_ALGO_AUTO: return "auto";
    case GBCONV_ALGO_DIRECT: return "direct";
    case GBCONV_ALGO_IGEMM_FFMA: return "igemm_ffma";
    case GBCONV_ALGO_IGEMM_TC: return "igemm_tc";
    case GBCONV_ALGO_DIRECT_TC: return "direct_tc";
    }
    return "unknown";
}

gbconv_status gbconv_check_device_error(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return GBCONV_ERR_CUDA;
    }
    unsigned int code = 0;
    if (read_and_clear_device_error(&code) != cudaSuccess) {
        cudaGetLastError();
        return GBCONV_ERR_CUDA;
    }
    return code ? GBCONV_ERR_TIMEOUT : GBCONV_OK;
}

gbconv_status gbconv_set_wait_limit_ns(uint64_t ns) {
    if (ns == 0) return GBCONV_ERR_SHAPE;
    set_wait_limit_ns(ns);
    return GBCONV_OK;
}

}  // extern "C"
