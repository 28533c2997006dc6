// Internal declarations shared by the host dispatcher and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "gbconv.h"

namespace gbconv {

// A validated problem with every derived extent. Index math is int64.
struct Problem {
    int ndim;                 // 2 or 3
    int N, C, D, H, W;        // D == 1 for 2D
    int OC, k, pad, stride;
    int kd;                   // kernel extent along D: k for 3D, 1 for 2D
    int pad_d;                // zero frames before D (front): pad, k-1 (causal) or 0; 0 for 2D
    int pad_d_back;           // zero frames after D
    int OD, OH, OW;
    int dtype, act, w_layout, algo;   // algo resolved (never AUTO)
    int taps;                 // kd * k * k
    int64_t x_elems, w_elems, y_elems;
    int64_t out_vol;          // OD * OH * OW (convolution output)
    int pool;                 // 1: 2x2 stride-2 max pool fused after the activation
    int cl;                   // 1: channels-last x [N][D][H][W][C] and y [N][OD][OH][OW][OC]
    int YH, YW;               // stored output rows / columns (OH/2, OW/2 when pooled)
    int64_t in_vol;           // D * H * W
    int elt;                  // bytes per stored element
};

// The tensor-core path can read channels-last 16-bit x in place: 16-byte rows.
inline bool tc_cl_direct(const Problem &p) { return p.cl && p.dtype != GBCONV_F32 && p.C % 8 == 0; }
// Tensor-core path channel padding: channels-last copies and packed weights
// carry C rounded up to a multiple of 8 (16-byte rows for TMA).
inline int tc_cpad(int C) { return (C + 7) / 8 * 8; }
// fp32 on the tensor cores (three TF32 products): x and the packed weights
// carry a hi and a lo half of Cs = C rounded up to 32 channels each (one
// 128-byte K block per 32 channels), so a row holds 2 * Cs channels.
inline int tc_split_half(int C) { return (C + 31) / 32 * 32; }
// Channels of one staged row of x / of packed weights on the tensor-core path.
inline int tc_row_channels(const Problem &p) {
    return p.dtype == GBCONV_F32 ? 2 * tc_split_half(p.C) : tc_cpad(p.C);
}
// CUDA-core implicit GEMM packs OC rounded up to this multiple.
constexpr int kFfmaOcAlign = 128;
inline int ffma_ocpad(int OC) { return (OC + kFfmaOcAlign - 1) / kFfmaOcAlign * kFfmaOcAlign; }

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Packed-weight bytes for the resolved algorithm.
size_t packed_weight_bytes(const Problem &p);
// Workspace layout for the resolved algorithm (offsets are 256-B aligned).
struct Workspace {
    size_t x_off = 0, x_bytes = 0;   // channels-last x (tensor-core path)
    size_t w_off = 0, w_bytes = 0;   // packed weights (when w_layout == OIHW)
    size_t part_off = 0, part_bytes = 0;   // split-K partial sums (fp32 CUDA-core GEMM)
    size_t total = 0;
};
// fp32 CUDA-core GEMM split over K (few tiles for the SMs): the partial-sum
// slices the workspace holds for it ([splits][OC][M] fp32), 0 when the layer
// does not qualify.
int ffma_split_slices(const Problem &p);
Workspace workspace_layout(const Problem &p);

// Whether a kernel family can run a problem (shared-memory and box limits).
bool direct_supported(const Problem &p);
bool stem_supported(const Problem &p);   // few-channel 3x3 direct kernel
bool tc_supported(const Problem &p);
bool stem_tc_supported(const Problem &p);   // fp32, 2D, k = 3, C <= 4, OC <= 128: tensor cores, split TF32

// Kernel launchers (each returns a cudaError_t from the launch).
cudaError_t launch_direct(const Problem &p, const void *x, const void *w_oihw,
                          const float *b, void *y, cudaStream_t s);
cudaError_t launch_direct_stem(const Problem &p, const void *x, const void *w_oihw,
                               const float *b, void *y, cudaStream_t s);
// part: room for `slices` fp32 partial-sum slices of [OC][M] (split-K), or
// null (no split).
cudaError_t launch_igemm_ffma(const Problem &p, const void *x,
                              const void *w_packed, const float *b, void *y,
                              float *part, int slices, cudaStream_t s);
cudaError_t launch_pack_ffma(const Problem &p, const void *w_oihw,
                             void *w_packed, cudaStream_t s);
cudaError_t launch_pack_tc(const Problem &p, const void *w_oihw,
                           void *w_packed, cudaStream_t s);
cudaError_t launch_to_channels_last(const Problem &p, const void *x,
                                    void *x_cl, cudaStream_t s);
// Both of the above in one launch (OIHW weights, x not read in place).
cudaError_t launch_prep_tc(const Problem &p, const void *w_oihw, void *w_packed,
                           const void *x, void *x_cl, cudaStream_t s);
cudaError_t launch_stem_tc(const Problem &p, const void *x, const void *w_oihw,
                           const float *b, void *y, cudaStream_t s);
// Returns cudaErrorInvalidValue when the tensor maps cannot be encoded.
cudaError_t launch_igemm_tc(const Problem &p, const void *x_cl,
                            const void *w_packed, const float *b, void *y,
                            cudaStream_t s);

// BatchNorm folded into OIHW weights and an fp32 bias (fold.cu).
cudaError_t launch_fold_bn(const Problem &p, const void *w, const float *b, const float *gamma,
                           const float *beta, const float *mean, const float *var, float eps,
                           void *w_out, float *b_out, cudaStream_t s);

// Launch with the programmatic stream-serialization attribute (the kernel
// calls pdl_wait() before its first global-memory access).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Status of a forward call from the error its launches returned: a CUDA
// call the library makes before launching (tensor-map encoding, attribute
// set-up) reports cudaErrorInvalidValue and maps to GBCONV_ERR_CUDA; any
// other launch error to GBCONV_ERR_LAUNCH (and is cleared).
inline gbconv_status launch_status(cudaError_t e) {
    if (e == cudaSuccess) return GBCONV_OK;
    if (e == cudaErrorInvalidValue) return GBCONV_ERR_CUDA;
    cudaGetLastError();
    return GBCONV_ERR_LAUNCH;
}

// Logging: with GBCONV_LOG=1 in the environment (read once per process)
// every forward call writes its kernel choice, and each launcher its launch
// geometry, as one line each to stderr. Host only; nothing is logged
// otherwise.
bool log_enabled();
void log_line(const char *fmt, ...) __attribute__((format(printf, 1, 2)));

// Device-side error word and wait limit (defined in igemm_tc.cu).
uint64_t wait_limit_ns();
void set_wait_limit_ns(uint64_t ns);
cudaError_t read_and_clear_device_error(unsigned int *code);

}  // namespace gbconv
