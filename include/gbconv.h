/*
 * gbconv: forward convolution (conv2d / conv3d, fused bias + ReLU) for one
 * NVIDIA GB300 (sm_103a), exposed as a plain C ABI.
 *
 * The operation (lpnh.cn/news/2745477, PP-OCR on Vulkan compute shaders,
 * section 2.2 "compute shader and SPIR-V"): every output element sums
 * input x weight over all input channels and kernel taps, with the input
 * coordinate derived from the output coordinate,
 *     i = o*stride - pad + tap      (per spatial axis),
 * taps outside the input contribute nothing (zero padding), and the bias of
 * the output channel is added last. It is cross-correlation (no kernel flip).
 * ReLU, when requested, is max(v, 0) applied after the bias, fused into the
 * write-back as in section 4.4 of the same page. Convolution3D adds a frame
 * (depth) axis with the same kernel size, pad and stride
 * (git.erdda.com/Tencent/ncnn/discussions/7001, SeedVR2 NCNN Vulkan,
 * section 3.2 "six custom layers").
 *
 * Output extent per axis: O = floor((I + 2*pad - k) / stride) + 1.
 *
 * Layouts (all densely packed, row-major, element offsets; x and y may
 * instead be channels-last, see GBCONV_FLAG_CHANNELS_LAST):
 *   x  conv2d [N][C][H][W]        conv3d [N][C][D][H][W]
 *   w  conv2d [OC][C][k][k]       conv3d [OC][C][k][k][k]   (w_layout OIHW)
 *      or the opaque packed form written by gbconv_weight_pack (w_layout PACKED)
 *   b  [OC], always float32, or NULL for no bias
 *   y  conv2d [N][OC][OH][OW]     conv3d [N][OC][OD][OH][OW]
 * x, w and y share the storage dtype (float32, float16 or bfloat16).
 * Arithmetic: float32 accumulation on every path; float16/bfloat16 results are
 * rounded to nearest-even from the float32 epilogue value.
 *
 * Ownership and memory: the caller owns every buffer (device memory). The
 * library allocates nothing: paths that need scratch space take it from the
 * caller's workspace (gbconv_workspace_size). x, w and b are read-only; y must
 * not overlap them or the workspace.
 *
 * Streams: calls enqueue work on the caller's stream and return without
 * synchronising; results are valid once the stream reaches that point. A
 * forward call makes no allocation, no synchronisation and no host read of
 * device data, so it can be recorded into a CUDA graph.
 *
 * Errors: every entry point returns a gbconv_status. Descriptors are validated
 * completely (an unknown activation, dtype, layout or algorithm, a non-zero
 * reserved field, a bad size, a NULL or misaligned pointer, overlapping
 * buffers, a short workspace) before any CUDA call; a rejected call has no side
 * effect. Nothing aborts the process.
 */
#ifndef GBCONV_H
#define GBCONV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gbconv_status {
    GBCONV_OK = 0,
    GBCONV_ERR_NULL = 1,               /* a required pointer is NULL */
    GBCONV_ERR_SHAPE = 2,              /* non-positive / oversized dims, empty output */
    GBCONV_ERR_DTYPE = 3,              /* unknown storage dtype */
    GBCONV_ERR_ACT = 4,                /* unknown activation */
    GBCONV_ERR_ALIGN = 5,              /* pointer not aligned to its element size */
    GBCONV_ERR_WORKSPACE = 6,          /* workspace missing, short or not 256-byte aligned */
    GBCONV_ERR_UNSUPPORTED_DEVICE = 7, /* current device is not compute capability 10.3 */
    GBCONV_ERR_LAUNCH = 8,             /* a kernel launch failed (cudaGetLastError) */
    GBCONV_ERR_TIMEOUT = 9,            /* a bounded device-side wait ran out */
    GBCONV_ERR_ALGO = 10,              /* unknown algorithm, or the forced one cannot run this shape */
    GBCONV_ERR_LAYOUT = 11,            /* unknown weight layout */
    GBCONV_ERR_OVERLAP = 12,           /* y overlaps x, w, b or the workspace, or the workspace x, w or b */
    GBCONV_ERR_CUDA = 13,              /* another CUDA runtime/driver call failed */
    GBCONV_ERR_RESERVED = 14,          /* a reserved flag bit is set, or an unknown frame-padding mode */
    GBCONV_ERR_TOO_LARGE = 15          /* gbconv_conv_fwd_noalloc: scratch need exceeds its fixed array */
} gbconv_status;

typedef enum gbconv_dtype {
    GBCONV_F32 = 0,
    GBCONV_F16 = 1,
    GBCONV_BF16 = 2
} gbconv_dtype;

typedef enum gbconv_act {
    GBCONV_ACT_NONE = 0,
    GBCONV_ACT_RELU = 1
} gbconv_act;

typedef enum gbconv_wlayout {
    GBCONV_W_OIHW = 0,     /* [OC][C][k][k] or [OC][C][k][k][k] */
    GBCONV_W_PACKED = 1    /* written by gbconv_weight_pack for the same desc */
} gbconv_wlayout;

/* Kernel families. AUTO picks by shape and dtype (see gbconv_select_algo). */
typedef enum gbconv_algo {
    GBCONV_ALGO_AUTO = 0,
    GBCONV_ALGO_DIRECT = 1,      /* direct, shared-memory halo + register micro-tile (small IC*k^d) */
    GBCONV_ALGO_IGEMM_FFMA = 2,  /* implicit GEMM on CUDA cores, exact fp32 FMA */
    GBCONV_ALGO_IGEMM_TC = 3,    /* implicit GEMM on tcgen05 tensor cores: fp16/bf16 storage (kind::f16), or
                                    fp32 storage as three TF32 products x_hi w_hi + x_lo w_hi + x_hi w_lo
                                    (kind::tf32, fp32 accumulate; relative error near 2^-20 per product,
                                    and a whole-output relative L2 error that grows with the reduction
                                    length C * k^d: measured at most 7.2e-6 up to 1,000 products, up to
                                    1.6e-5 beyond, so AUTO takes it for fp32 only up to 1,000) */
    GBCONV_ALGO_DIRECT_TC = 4    /* fp32, 2D, k = 3, C <= 4, OC <= 128 (image stems) on tcgen05 tensor
                                    cores: x and w split into TF32 hi + lo parts, one MMA chain forms
                                    (x_hi + x_lo) * w_hi and (x_hi + x_lo) * w_lo, fp32 accumulate;
                                    relative error near 2^-20 per product */
} gbconv_algo;

/*
 * Padding of the frame axis of conv3d (bits 0-1 of gbconv_desc.flags). The
 * video VAE of git.erdda.com/Tencent/ncnn/discussions/7001 (SeedVR2, section
 * 3.3) runs causal Convolution3D: an output frame sees only its own and
 * earlier input frames, the missing leading frames being zeros on the first
 * chunk and the previous chunk's last k-1 frames afterwards.
 *   SYMMETRIC: `pad` zero frames before and after (the same as H and W).
 *   CAUSAL:    k-1 zero frames before, none after; output frame t reads input
 *              frames t*stride-(k-1) .. t*stride. OD = floor((D-1)/stride)+1.
 *   NONE:      no frame padding (for callers that prepend the k-1 cached frames
 *              of the previous chunk themselves). OD = floor((D-k)/stride)+1.
 * H and W are always padded by `pad` on both sides. conv2d takes SYMMETRIC only.
 */
typedef enum gbconv_tpad {
    GBCONV_TPAD_SYMMETRIC = 0,
    GBCONV_TPAD_CAUSAL = 1,
    GBCONV_TPAD_NONE = 2
} gbconv_tpad;
#define GBCONV_FLAG_TPAD_MASK 0x3
/*
 * Bit 2 of gbconv_desc.flags: a 2x2, stride-2 max pool fused into the
 * epilogue after bias and activation (floor mode: y is [N][OC][OH/2][OW/2];
 * a last odd row / column is dropped), as lpnh.cn/news/2745477 section 4.4
 * fuses conv, ReLU and pooling into one shader for small-channel layers.
 * conv2d only, on the direct few-channel 3x3 kernel (C <= 4, stride 1 or 2,
 * pad <= 1); other shapes or algorithms return GBCONV_ERR_ALGO.
 */
#define GBCONV_FLAG_MAXPOOL2 0x4
/*
 * Bit 3 of gbconv_desc.flags: channels-last activations. x is
 * [N][H][W][C] (conv2d) or [N][D][H][W][C] (conv3d) and y is
 * [N][OH][OW][OC] or [N][OD][OH][OW][OC]; weights keep their layout (OIHW /
 * OIDHW or packed). With channels-last output feeding channels-last input,
 * convolutions chain with no re-layout between them, the way
 * git.erdda.com/Tencent/ncnn/discussions/7001 (SeedVR2, limitations and
 * roadmap) plans to keep its packed channel layout across the video-VAE's
 * layers; lpnh.cn/news/2745477 section 2.3 weighs NHWC's vector-friendly
 * channel runs against NCHW's simplicity.
 * Kernels: the tensor-core implicit GEMM (float16/bfloat16 with C a multiple
 * of 8 and x 16-byte aligned: it reads x in place, so the call needs no
 * channels-last copy in the workspace; float32: x is split into its TF32
 * halves in the workspace as for NCHW input) and the CUDA-core implicit GEMM
 * (any dtype and C). AUTO picks the first when it applies, else the second;
 * the direct kernels and the fused max pool return GBCONV_ERR_ALGO.
 */
#define GBCONV_FLAG_CHANNELS_LAST 0x8

/*
 * Problem descriptor. Zero-initialise it, then set every field you use.
 * Kernel size, pad and stride are the same on every spatial axis (the pages'
 * single kSize/pad/stride parameters); conv3d's frame axis may instead be
 * padded causally (flags). For conv2d, D must be 1.
 */
typedef struct gbconv_desc {
    int N, C, D, H, W;        /* input: batch, channels, frames (1 for 2D), height, width */
    int OC, k, pad, stride;   /* output channels, kernel size, zero pad, stride */
    int dtype;                /* gbconv_dtype: storage type of x, w, y */
    int act;                  /* gbconv_act */
    int w_layout;             /* gbconv_wlayout */
    int algo;                 /* gbconv_algo */
    int flags;                /* bits 0-1: gbconv_tpad (conv3d frame padding); bit 2: fused 2x2 max
                                 pool; bit 3: channels-last x and y; other bits must be 0 */
    void *workspace;          /* device scratch, >= gbconv_workspace_size bytes, 256-B aligned */
    size_t workspace_bytes;
} gbconv_desc;

/* Limits enforced by validation. */
#define GBCONV_MAX_DIM 65535      /* any of N, C, D, H, W, OC */
#define GBCONV_MAX_K 16           /* kernel size */
#define GBCONV_MAX_STRIDE 8
#define GBCONV_MAX_ELEMS ((int64_t)1 << 36)   /* elements of x, w or y */

/*
 * Forward convolution, 2D. x, w, y: device pointers in the layouts above,
 * aligned to their element size; b: device float32 [OC] or NULL. Enqueued on
 * `stream`; returns before the work runs.
 */
gbconv_status gbconv_conv2d_fwd(const gbconv_desc *desc, const void *x,
                                const void *w, const float *b, void *y,
                                cudaStream_t stream);

/* Forward convolution, 3D (Convolution3D over frames). Same contract. */
gbconv_status gbconv_conv3d_fwd(const gbconv_desc *desc, const void *x,
                                const void *w, const float *b, void *y,
                                cudaStream_t stream);

/* Output extents for ndim = 2 (OD = 1) or 3. Host only, no CUDA call. */
gbconv_status gbconv_output_shape(const gbconv_desc *desc, int ndim, int *OD,
                                  int *OH, int *OW);

/*
 * Bytes of caller workspace the forward call needs for this desc (0 when the
 * chosen kernel needs none). Scratch holds the re-laid-out input (tensor-core
 * path: channels-last copy of x; for float32, x split into TF32 hi and lo
 * halves), with w_layout OIHW the packed weights, and, for a float32 layer on
 * the CUDA-core implicit GEMM (C a multiple of 16, NC(D)HW x) with fewer
 * than 160 tiles of 128 pixels x 128 output channels, the fp32 partial sums
 * of its split over K (at most 8 slices of OC x N x OD x OH x OW, 64 MB at
 * most). Host only.
 */
gbconv_status gbconv_workspace_size(const gbconv_desc *desc, int ndim,
                                    size_t *bytes);

/* Bytes of the packed weight buffer for this desc. Host only. */
gbconv_status gbconv_weight_packed_size(const gbconv_desc *desc, int ndim,
                                        size_t *bytes);

/*
 * Re-lay OIHW/OIDHW weights once into the form the chosen kernel reads, so
 * that later calls can pass w_layout = PACKED and skip the per-call packing
 * (the weights are re-arranged at export time, not in the hot path:
 * lpnh.cn/news/2745477 sections 2.3 and 4.2). A pure permutation plus zero
 * padding; bit-exact. w_packed must hold gbconv_weight_packed_size bytes and be
 * 256-byte aligned. The packed form is only valid for a desc that selects the
 * same algorithm, dtype, C, OC, k and ndim.
 */
gbconv_status gbconv_weight_pack(const gbconv_desc *desc, int ndim,
                                 const void *w_oihw, void *w_packed,
                                 cudaStream_t stream);

/*
 * Fold an inference-mode BatchNorm that follows the convolution into its
 * weights and bias (lpnh.cn/news/2745477 section 3.1: BN folded into the
 * conv at export, so the graph runs one conv). For each output channel oc,
 * s = gamma[oc] / sqrt(var[oc] + eps) (fp32), and
 *     w_out[oc][...] = w[oc][...] * s      (rounded to the storage dtype)
 *     b_out[oc]      = (b[oc] - mean[oc]) * s + beta[oc]   (b may be NULL: 0)
 * so a forward call with (w_out, b_out) computes
 * gamma * (conv(x, w, b) - mean) / sqrt(var + eps) + beta (ReLU, if set in the
 * desc, still applies after). w / w_out: OIHW/OIDHW in the desc's dtype,
 * aligned to the element size; b, gamma, beta, mean, var, b_out: device
 * float32 [OC]. w_out may equal w (in place) and b_out may equal b; no other
 * overlap. eps must be finite and >= 0. Enqueued on `stream`.
 * Errors: validation codes as for the forward call; GBCONV_ERR_NULL for a
 * missing gamma/beta/mean/var/w/w_out/b_out; GBCONV_ERR_SHAPE for a bad eps;
 * GBCONV_ERR_LAUNCH if the launch fails.
 */
gbconv_status gbconv_fold_batchnorm(const gbconv_desc *desc, int ndim, const void *w,
                                    const float *b, const float *gamma, const float *beta,
                                    const float *mean, const float *var, float eps,
                                    void *w_out, float *b_out, cudaStream_t stream);

/* The algorithm a forward call with this desc runs (resolves AUTO). Host only. */
gbconv_status gbconv_select_algo(const gbconv_desc *desc, int ndim, int *algo);

/* 1 if `device` is a compute capability 10.3 GPU this library can run on, else 0.
   Never aborts, also on a machine without a GPU (cf. the backend-valid query
   of githubissues.com/ysh329/OpenCL-101/52, "init fault tolerance"). */
int gbconv_device_supported(int device);

/* Static, human-readable name of a status / an algorithm. Never NULL. */
const char *gbconv_status_string(gbconv_status status);
const char *gbconv_algo_name(int algo);

/*
 * Synchronise `stream`, then read and clear the library's device error word
 * for the current device. Returns GBCONV_ERR_TIMEOUT if a bounded wait inside
 * a tensor-core kernel ran out since the last check (that kernel stopped
 * early and its output is undefined), GBCONV_OK otherwise. Not for use inside
 * stream capture.
 */
gbconv_status gbconv_check_device_error(cudaStream_t stream);

/*
 * Upper bound, in nanoseconds, on any single device-side wait inside the
 * tensor-core kernel (default 2e9). Host only; affects later launches.
 */
gbconv_status gbconv_set_wait_limit_ns(uint64_t ns);

/*
 * Forward convolution that allocates nothing and takes no workspace.
 * The pages have no counterpart of this entry point; it is a service for
 * callers that cannot obtain device memory themselves, e.g. code running
 * while a stream is being captured into a CUDA graph (where cudaMalloc is
 * not allowed), real-time loops that must never enter the allocator, or
 * plain-C hosts without a caching allocator.
 *
 * It runs the CUDA-core implicit-GEMM path (any dtype, 2D or 3D by `ndim`)
 * and keeps that path's only scratch, the packed weights, in a fixed device
 * array inside the library of GBCONV_NOALLOC_SCRATCH_BYTES bytes, which every
 * GPU that loads the library holds until the process exits.
 *   desc      as for gbconv_conv2d_fwd; algo must be AUTO or IGEMM_FFMA,
 *             w_layout must be OIHW, workspace fields are ignored.
 *   x, w, b, y  caller-owned device pointers, as for gbconv_conv2d_fwd.
 * Errors: the validation codes of gbconv_conv2d_fwd, except that the fused
 * 2x2 max pool (flags bit 2), which only the direct kernel has, is always
 * GBCONV_ERR_ALGO here; GBCONV_ERR_TOO_LARGE when the packed weights
 * (taps * C * roundup(OC, 128) elements of the storage type) exceed the
 * fixed array; GBCONV_ERR_CUDA / GBCONV_ERR_LAUNCH as for the forward call.
 * All calls on a device share the array: calls whose kernels overlap on the
 * GPU race, so serialise them on one stream. The array keeps the last call's
 * contents; every call rewrites all of it that it reads. The first call on a
 * device looks up the array's address (cudaGetSymbolAddress, that device
 * current); make that first call before any stream capture. That address is
 * cached for the life of the device's primary context: after cudaDeviceReset
 * the process must not call this entry point again.
 */
#define GBCONV_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
gbconv_status gbconv_conv_fwd_noalloc(const gbconv_desc *desc, int ndim,
                                      const void *x, const void *w,
                                      const float *b, void *y,
                                      cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* GBCONV_H */
