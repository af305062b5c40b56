// Shared helpers of the CUDA library: element loads/stores with fp32
// conversion, warp reductions, the workspace header and host-side checks.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "tee.h"

namespace tee {

// ------------------------------------------------------------ workspace header
// Word 0: first device fault code (TEE_DEVERR_*), word 1: its detail.
// Words 8..63: counters of "last block" reductions, left at zero by every call.
enum { WS_ERR = 0, WS_DETAIL = 1, WS_CNT_GATE = 8, WS_CNT_ROUTER = 9 };

__device__ __forceinline__ void record_fault(void* ws, int code, int detail) {
    int32_t* h = reinterpret_cast<int32_t*>(ws);
    if (atomicCAS(h + WS_ERR, 0, code) == 0) h[WS_DETAIL] = detail;
}

__host__ __device__ __forceinline__ uint32_t* ws_counter(void* ws, int idx) {
    return reinterpret_cast<uint32_t*>(ws) + idx;
}

template <typename T>
__host__ __device__ __forceinline__ T* ws_at(void* ws, size_t byte_off) {
    return reinterpret_cast<T*>(reinterpret_cast<char*>(ws) + byte_off);
}

// ------------------------------------------------------------ element access
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ void unpack_bf16x2(uint32_t u, float& lo, float& hi) {
    lo = __uint_as_float(u << 16);
    hi = __uint_as_float(u & 0xFFFF0000u);
}
__device__ __forceinline__ void unpack_f16x2(uint32_t u, float& lo, float& hi) {
    __half2 h = *reinterpret_cast<__half2*>(&u);
    float2 f = __half22float2(h);
    lo = f.x;
    hi = f.y;
}

// Eight consecutive elements (16-byte aligned for 2-byte types, 32 for fp32).
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&f)[8]) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    unpack_bf16x2(u.x, f[0], f[1]);
    unpack_bf16x2(u.y, f[2], f[3]);
    unpack_bf16x2(u.z, f[4], f[5]);
    unpack_bf16x2(u.w, f[6], f[7]);
}
__device__ __forceinline__ void load8(const __half* p, float (&f)[8]) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    unpack_f16x2(u.x, f[0], f[1]);
    unpack_f16x2(u.y, f[2], f[3]);
    unpack_f16x2(u.z, f[4], f[5]);
    unpack_f16x2(u.w, f[6], f[7]);
}
__device__ __forceinline__ void load8(const float* p, float (&f)[8]) {
    float4 a = __ldg(reinterpret_cast<const float4*>(p));
    float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&f)[8]) {
    uint4 u = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                         pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
    *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ void store8(__half* p, const float (&f)[8]) {
    uint4 u = make_uint4(pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]),
                         pack_f16x2(f[4], f[5]), pack_f16x2(f[6], f[7]));
    *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ void store8(float* p, const float (&f)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}

// Copy nv 16-byte vectors by one warp, eight loads per lane in flight.
__device__ __forceinline__ void warp_copy16(uint4* __restrict__ dst, const uint4* __restrict__ src, int nv,
                                            int lane) {
    constexpr int U = 8;
    for (int k0 = lane; k0 < nv; k0 += 32 * U) {
        uint4 t[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (k0 + 32 * u < nv) t[u] = __ldg(src + k0 + 32 * u);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (k0 + 32 * u < nv) dst[k0 + 32 * u] = t[u];
    }
}

// ------------------------------------------------------------ dependent launches
// Let a kernel enqueued after this one with programmatic stream serialization
// start now; it waits for this grid to complete before reading what it writes.
__device__ __forceinline__ void allow_dependents() {
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// In a kernel launched with programmatic stream serialization: wait until the
// kernel enqueued before it has completed and its writes are visible (returns
// at once otherwise).
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------ reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ unsigned warp_sum_u(unsigned v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Exit decision shared by both gates: strict score > threshold in fp32.
__device__ __forceinline__ uint8_t exits(float s, float thr) { return s > thr ? 1 : 0; }

// "Last block" batch flag: each block publishes the minimum score it saw;
// the block that arrives last reduces them, writes the all-tokens flag and,
// under the batch rule, broadcasts it into the mask. Needs no spin wait.
static __device__ __noinline__ void batch_flag_tail(float block_min, int n, float thr, int rule,
                                uint8_t* mask, int32_t* flag, float* ws_mins, uint32_t* counter) {
    __shared__ int s_last;
    __shared__ float s_red[32];
    if (threadIdx.x == 0) {
        ws_mins[blockIdx.x] = block_min;
        __threadfence();
        unsigned prev = atomicAdd(counter, 1u);
        s_last = (prev == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    float m = INFINITY;
    for (unsigned i = threadIdx.x; i < gridDim.x; i += blockDim.x)
        m = fminf(m, *reinterpret_cast<volatile float*>(ws_mins + i));
    m = warp_min(m);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < (blockDim.x >> 5) ? s_red[threadIdx.x] : INFINITY;
        v = warp_min(v);
        if (threadIdx.x == 0) s_red[0] = v;
    }
    __syncthreads();
    const uint8_t f = (n > 0 && s_red[0] > thr) ? 1 : 0;
    if (threadIdx.x == 0) {
        if (flag) *flag = f;
        *counter = 0u;
    }
    if (rule == TEE_RULE_BATCH_ALL)
        for (int t = threadIdx.x; t < n; t += blockDim.x) mask[t] = f;
}


// ------------------------------------------------------------ host side
tee_status cuda_status(cudaError_t e);
// Status of the launch just made; also counts it (tee_launch_count).
tee_status launch_status();
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t dtype_bytes(int dt) { return dt == TEE_F32 ? 4 : (dt == TEE_F16 || dt == TEE_BF16) ? 2 : 0; }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int sm_count();

}  // namespace tee
