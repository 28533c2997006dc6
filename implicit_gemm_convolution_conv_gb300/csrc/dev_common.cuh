// Device helpers shared by all kernels: storage-type conversion and the fused
// epilogue (bias, optional ReLU, rounding to the storage type).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace gbconv {

template <typename T> struct Storage;
template <> struct Storage<float> {
    using Pair = float2;
    static __device__ __forceinline__ Pair pack2(float lo, float hi) { return make_float2(lo, hi); }
    static __device__ __forceinline__ float load(const float *p) { return __ldg(p); }
    static __device__ __forceinline__ float to_float(float v) { return v; }
    static __device__ __forceinline__ float from_float(float v) { return v; }
};
template <> struct Storage<__half> {
    using Pair = __half2;
    static __device__ __forceinline__ Pair pack2(float lo, float hi) { return __floats2half2_rn(lo, hi); }
    static __device__ __forceinline__ float load(const __half *p) { return __half2float(__ldg(p)); }
    static __device__ __forceinline__ float to_float(__half v) { return __half2float(v); }
    static __device__ __forceinline__ __half from_float(float v) { return __float2half_rn(v); }
};
template <> struct Storage<__nv_bfloat16> {
    using Pair = __nv_bfloat162;
    static __device__ __forceinline__ Pair pack2(float lo, float hi) { return __floats2bfloat162_rn(lo, hi); }
    static __device__ __forceinline__ float load(const __nv_bfloat16 *p) { return __bfloat162float(__ldg(p)); }
    static __device__ __forceinline__ float to_float(__nv_bfloat16 v) { return __bfloat162float(v); }
    static __device__ __forceinline__ __nv_bfloat16 from_float(float v) { return __float2bfloat16_rn(v); }
};

// Programmatic dependent launch. Kernels are launched with the programmatic
// stream-serialization attribute, so a kernel may begin (launch, shared
// memory and TMEM set-up) while the previous kernel in the stream is still
// finishing. Every thread waits for the previous kernel to complete, and its
// writes to be visible, before its first access to global memory; each
// kernel allows its successor to launch as soon as it has started. Without
// the attribute both instructions do nothing.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Fused epilogue (lpnh.cn/news/2745477 section 2.2: bias added at write-back;
// section 4.4: ReLU fused into the same write): v = acc + b, then max(v, 0).
__device__ __forceinline__ float epilogue(float acc, float bias, int relu) {
    float v = acc + bias;
    return relu ? fmaxf(v, 0.0f) : v;
}

}  // namespace gbconv
