// BatchNorm folded into the convolution's weights and bias.
//
// lpnh.cn/news/2745477 section 3.1 folds the BatchNorm that follows a
// convolution into that convolution when the model is exported, so the
// inference graph runs one conv instead of conv + BN. For output channel oc,
// with s = gamma[oc] / sqrt(var[oc] + eps):
//     w'[oc][...] = w[oc][...] * s
//     b'[oc]      = (b[oc] - mean[oc]) * s + beta[oc]      (b = 0 when absent)
// so that conv(x, w', b') = gamma * (conv(x, w, b) - mean) / sqrt(var + eps) + beta.
// The scale is formed in fp32; w' is rounded to the storage type (RN-even).
#include "dev_common.cuh"
#include "internal.h"

namespace gbconv {
namespace {

template <typename T>
__global__ void fold_bn_kernel(const T *__restrict__ w, const float *__restrict__ b,
                               const float *__restrict__ gamma, const float *__restrict__ beta,
                               const float *__restrict__ mean, const float *__restrict__ var,
                               float eps, T *__restrict__ w_out, float *__restrict__ b_out,
                               int OC, int64_t per_oc) {
    const int oc = blockIdx.y;
    const float s = gamma[oc] / sqrtf(var[oc] + eps);
    const T *src = w + (int64_t)oc * per_oc;
    T *dst = w_out + (int64_t)oc * per_oc;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < per_oc;
         i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = Storage<T>::from_float(Storage<T>::to_float(src[i]) * s);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        const float bb = b ? b[oc] : 0.0f;
        b_out[oc] = (bb - mean[oc]) * s + beta[oc];
    }
}

template <typename T>
cudaError_t launch_fold_t(const Problem &p, const void *w, const float *b, const float *gamma,
                          const float *beta, const float *mean, const float *var, float eps,
                          void *w_out, float *b_out, cudaStream_t s) {
    const int64_t per_oc = (int64_t)p.C * p.taps;
    const int64_t blocks = (per_oc + 255) / 256;
    dim3 grid((unsigned)(blocks < 64 ? blocks : 64), (unsigned)p.OC);
    fold_bn_kernel<T><<<grid, 256, 0, s>>>(static_cast<const T *>(w), b, gamma, beta, mean, var, eps,
                                           static_cast<T *>(w_out), b_out, p.OC, per_oc);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fold_bn(const Problem &p, const void *w, const float *b, const float *gamma,
                           const float *beta, const float *mean, const float *var, float eps,
                           void *w_out, float *b_out, cudaStream_t s) {
    switch (p.dtype) {
    case GBCONV_F32: return launch_fold_t<float>(p, w, b, gamma, beta, mean, var, eps, w_out, b_out, s);
    case GBCONV_F16: return launch_fold_t<__half>(p, w, b, gamma, beta, mean, var, eps, w_out, b_out, s);
    default: return launch_fold_t<__nv_bfloat16>(p, w, b, gamma, beta, mean, var, eps, w_out, b_out, s);
    }
}

}  // namespace gbconv
