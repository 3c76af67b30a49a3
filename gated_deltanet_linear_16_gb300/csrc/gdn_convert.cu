// gdn_convert.cu -- h-state dtype converters, binary32 <-> binary16.
//
// Follows metrale_model_layers/layers/ops/ssm_gdn_a.rs, launchers
// `ssm_h_state_f32_to_f16` (round to nearest even) and
// `ssm_h_state_f16_to_f32` (exact widening): n elements, grid-stride, source
// and destination must not alias.
//
// Pure HBM streams (6 bytes per element either way).  The vector kernels move
// 4 elements per thread per step -- one 16-byte fp32 vector <-> one 8-byte
// fp16 vector -- so every warp-wide load and store covers one contiguous span
// (512 B of fp32, 256 B of fp16) and no store leaves part of a sector for a
// later instruction; 32 steps are in flight per thread.  The grid is a whole
// number of waves (8 CTAs of 256 threads per SM), and the few elements past
// the last full vector are done by the first threads.  Unaligned pointers take
// a scalar grid-stride kernel with the same results.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 8;   // 8: f32 -> f16 183-187 us over the 202 M-element pool, 4: 189; f16 -> f32 alike
constexpr int kUnroll = 32;   // steps in flight per thread: 8 -> 32 took f16 -> f32 from 203 to 190 us

__device__ __forceinline__ unsigned pack_h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<unsigned *>(&h);
}
__device__ __forceinline__ float2 unpack_h2(unsigned u) {
    __half2 h = *reinterpret_cast<__half2 *>(&u);
    return __half22float2(h);
}

__global__ void __launch_bounds__(kThreads)
f32_to_f16_vec(const float *__restrict__ src, uint16_t *__restrict__ dst, uint64_t n)
{
    const uint64_t nvec = n / 4;
    const uint64_t stride = (uint64_t)gridDim.x * kThreads;
    const uint64_t tid = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
    uint2 *d2 = reinterpret_cast<uint2 *>(dst);
    uint64_t i = tid;
    for (; i + (kUnroll - 1) * stride < nvec; i += kUnroll * stride) {
        uint4 a[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) a[u] = __ldcs(s4 + i + u * stride);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            __stcs(d2 + i + u * stride, make_uint2(pack_h2(__uint_as_float(a[u].x), __uint_as_float(a[u].y)),
                                                   pack_h2(__uint_as_float(a[u].z), __uint_as_float(a[u].w))));
    }
    for (; i < nvec; i += stride) {
        const uint4 a = __ldcs(s4 + i);
        __stcs(d2 + i, make_uint2(pack_h2(__uint_as_float(a.x), __uint_as_float(a.y)),
                                  pack_h2(__uint_as_float(a.z), __uint_as_float(a.w))));
    }
    const uint64_t tail = nvec * 4 + tid;
    if (tail < n) {
        __half h = __float2half_rn(src[tail]);
        dst[tail] = *reinterpret_cast<uint16_t *>(&h);
    }
}

__global__ void __launch_bounds__(kThreads)
f16_to_f32_vec(const uint16_t *__restrict__ src, float *__restrict__ dst, uint64_t n)
{
    const uint64_t nvec = n / 4;
    const uint64_t stride = (uint64_t)gridDim.x * kThreads;
    const uint64_t tid = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
    const uint2 *s2 = reinterpret_cast<const uint2 *>(src);
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
    uint64_t i = tid;
    for (; i + (kUnroll - 1) * stride < nvec; i += kUnroll * stride) {
        uint2 a[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) a[u] = __ldcs(s2 + i + u * stride);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const float2 x0 = unpack_h2(a[u].x), x1 = unpack_h2(a[u].y);
            __stcs(d4 + i + u * stride, make_uint4(__float_as_uint(x0.x), __float_as_uint(x0.y),
                                                   __float_as_uint(x1.x), __float_as_uint(x1.y)));
        }
    }
    for (; i < nvec; i += stride) {
        const uint2 a = __ldcs(s2 + i);
        const float2 x0 = unpack_h2(a.x), x1 = unpack_h2(a.y);
        __stcs(d4 + i, make_uint4(__float_as_uint(x0.x), __float_as_uint(x0.y),
                                  __float_as_uint(x1.x), __float_as_uint(x1.y)));
    }
    const uint64_t tail = nvec * 4 + tid;
    if (tail < n) {
        __half h = *reinterpret_cast<const __half *>(src + tail);
        dst[tail] = __half2float(h);
    }
}

__global__ void __launch_bounds__(kThreads)
f32_to_f16_scalar(const float *__restrict__ src, uint16_t *__restrict__ dst, uint64_t n)
{
    const uint64_t stride = (uint64_t)gridDim.x * kThreads;
    for (uint64_t i = (uint64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += stride) {
        __half h = __float2half_rn(src[i]);
        dst[i] = *reinterpret_cast<uint16_t *>(&h);
    }
}

__global__ void __launch_bounds__(kThreads)
f16_to_f32_scalar(const uint16_t *__restrict__ src, float *__restrict__ dst, uint64_t n)
{
    const uint64_t stride = (uint64_t)gridDim.x * kThreads;
    for (uint64_t i = (uint64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += stride) {
        __half h = *reinterpret_cast<const __half *>(src + i);
        dst[i] = __half2float(h);
    }
}

unsigned grid_for(uint64_t work_items)
{
    // whole waves of kCtasPerSm CTAs per SM, never more CTAs than work
    const uint64_t full = (uint64_t)sm_count() * kCtasPerSm;
    const uint64_t need = (work_items + kThreads - 1) / kThreads;
    const uint64_t g = need < full ? need : full;
    return (unsigned)(g > 0 ? g : 1);
}

}  // namespace

cudaError_t launch_f32_to_f16(const float *src, uint16_t *dst, uint64_t n, bool vec, cudaStream_t s)
{
    if (vec) f32_to_f16_vec<<<grid_for(n / 4 > 0 ? n / 4 : n), kThreads, 0, s>>>(src, dst, n);
    else f32_to_f16_scalar<<<grid_for(n), kThreads, 0, s>>>(src, dst, n);
    return cudaGetLastError();
}

cudaError_t launch_f16_to_f32(const uint16_t *src, float *dst, uint64_t n, bool vec, cudaStream_t s)
{
    if (vec) f16_to_f32_vec<<<grid_for(n / 4 > 0 ? n / 4 : n), kThreads, 0, s>>>(src, dst, n);
    else f16_to_f32_scalar<<<grid_for(n), kThreads, 0, s>>>(src, dst, n);
    return cudaGetLastError();
}

}  // namespace gdn
