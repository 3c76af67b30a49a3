// gdn_internal.cuh -- parameter blocks, launcher declarations and small device
// helpers shared by the libgdn translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>
#include <utility>

namespace gdn {

constexpr unsigned kFull = 0xffffffffu;

// Everything one decode launch needs.  Pointers are device pointers; strides
// and the pitch are in elements of their own arrays.
struct DecodeParams {
    void *state;            // float* or __half*
    int64_t pitch;          // state elements between sequence slots
    const float *q, *k, *v, *alpha, *beta;
    const float *z, *gn;    // norm variant only
    float *o;               // raw variant only
    uint16_t *out;          // norm variant only (bf16 bits)
    int64_t qk_stride, v_stride, gb_stride, z_stride, o_stride, out_stride;
    int batch, nk, nv, d;
    float eps;
    float inv_sqrt_d;       // 1/sqrt(D) rounded once on the host
    // two-token variant only: the state after the first token, slot pitch in elements.
    // Token rows are then b * 2 + t for q, k, v, alpha, beta and o.
    void *state_mid;
    int64_t mid_pitch;
    // int8 epilogue only: codes [batch][nv*d], group scales [batch][nv*d/32],
    // and (nullable) the fp32 normed values [batch][nv*d]; row strides in elements.
    int8_t *xq;
    float *xs, *y;
    int64_t xq_stride, xs_stride, y_stride;
    // set by the launcher: bytes of the CTA's state head an early-launched
    // kernel asks the L2 for while it waits (see early_start)
    unsigned pf_bytes;
};

// What the single-token kernels write after the step: raw o, the normed output
// as bf16, or the normed output as int8 groups of 32.
constexpr int kEpiRaw = 0, kEpiBf16 = 1, kEpiQ8 = 2;

// The gated RMS norm over rows of raw outputs (rows of NV heads x D values).
struct NormParams {
    const float *o, *z, *gn;
    uint16_t *out;                     // bf16 epilogue
    int8_t *xq;                        // int8 epilogue: codes, group scales, optional fp32 y
    float *xs, *y;
    int64_t rows, o_stride, z_stride, out_stride, xq_stride, xs_stride, y_stride;
    int nv, d;
    float eps;
};

struct PrefillParams {
    void *state;            // float* or __half*
    int64_t pitch;
    const float *q, *k, *v, *alpha, *beta;
    float *o;
    int64_t qk_stride, v_stride, gb_stride, o_stride;   // per token row
    int batch, seq_len, nk, nv, d;
    float inv_sqrt_d;
    unsigned zero;          // always 0; see prefill_d128 (orders shared loads)
};

// The fused decode from projections: conv ring update + silu, L2 of q/k,
// gates from logits, the recurrence and the gated norm.
struct ConvNormParams {
    void *state;
    int64_t pitch;
    float *ring;            // [batch] slots of taps * C, [tap][channel], newest tap last
    int64_t ring_pitch;
    const float *x;         // [batch] rows of C = 2*NK*D + NV*D: [q heads | k heads | v heads]
    int64_t x_stride;
    const float *w;         // [taps][C]
    const float *br, *ar;   // [batch] rows of NV gate logits
    int64_t gate_stride;
    const float *dt, *rate; // [NV]
    const float *z, *gn;
    uint16_t *out;
    int *counters;          // [batch * NK] readers of each key head's q/k ring rows; zero between calls
    int64_t z_stride, out_stride;
    int batch, nk, nv, d, taps, repeat;   // repeat = NV / NK value heads per key head
    float l2_eps, eps, inv_sqrt_d;
    unsigned pf_bytes;      // as DecodeParams::pf_bytes
};

// Launchers (one per translation unit family).  They pick the kernel variant
// (fast D == 128 path when the alignment allows it, general otherwise) and
// return the launch status.
cudaError_t launch_decode(const DecodeParams &p, bool f16_state, int epi, bool fast, cudaStream_t s);
cudaError_t launch_decode_chunk2(const DecodeParams &p, bool f16_state, bool fast, cudaStream_t s);
cudaError_t launch_prefill(const PrefillParams &p, bool f16_state, bool fast, cudaStream_t s);
cudaError_t launch_conv_norm(const ConvNormParams &p, bool f16_state, bool fast, cudaStream_t s);
cudaError_t launch_gate_norm(const NormParams &p, int epi, bool fast, cudaStream_t s);
cudaError_t launch_f32_to_f16(const float *src, uint16_t *dst, uint64_t n, bool vec, cudaStream_t s);
cudaError_t launch_f16_to_f32(const uint16_t *src, float *dst, uint64_t n, bool vec, cudaStream_t s);

// gdn_decode_conv_norm's argument checks and launch, shared by its two entry
// points.  `counters_of` null: `workspace` is the caller's counter buffer (an
// operand, checked like the others).  Otherwise `workspace` is ignored and the
// counters' address comes from counters_of, which runs only after every check
// has passed (a rejected or empty call makes no CUDA call).
using CountersFn = cudaError_t (*)(int32_t **);
int decode_conv_norm_entry(void *state, int state_dtype, int64_t state_pitch,
                           float *conv_state, int64_t conv_pitch, int taps,
                           const float *x, const float *conv_w,
                           const float *br, const float *ar, const float *dt, const float *rate,
                           const float *z, const float *gn, float l2_eps, float eps,
                           uint16_t *out, int32_t *workspace, CountersFn counters_of,
                           int batch, int nk, int nv, int d,
                           int64_t x_stride, int64_t gate_stride, int64_t z_stride,
                           int64_t out_stride, void *stream);

// Number of SMs of the current device (cached per device id).
int sm_count();

// GDN_OK for cudaSuccess; otherwise records e for gdn_last_cuda_error() on
// this host thread and returns GDN_ERR_CUDA.
int report_cuda_error(cudaError_t e);

// Raise kernel Kern's dynamic shared-memory limit to `bytes` (above the 48 KB
// default).  The attribute belongs to the current device's context, so it is
// set once per device (ids below 64; others every call).
template <auto Kern>
cudaError_t allow_dynamic_smem(int bytes)
{
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t{1} << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// Early launch.  A kernel launched with programmatic stream serialisation may
// become resident while the kernel before it in the stream drains its last
// CTAs, so its own start (and, with an L2 prefetch, its first state bytes)
// overlaps that drain.  Measured on GB300: a gain for grids of a few waves
// (one layer at batch 32: 3.4 waves, -4 to -6 % per launch with a quarter or
// half of the head prefetched), a loss for grids of many waves (the 256-slot
// fp16 pool: 20-27 waves, up to +3 % without a prefetch and +7 % with one),
// so it is taken for grids of at most kEarlyMaxWaves waves of `ctas_per_sm`
// CTAs per SM.
constexpr int kEarlyMaxWaves = 4;
inline bool early_grid(unsigned grid, int ctas_per_sm)
{
    return (int64_t)grid <= (int64_t)kEarlyMaxWaves * sm_count() * ctas_per_sm;
}

// Launch kern with programmatic stream serialisation when `early`, else as a
// plain launch.  `early` only for a kernel instantiated with early_start<true>.
template <typename... KArgs, typename... Args>
cudaError_t launch_early(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t s,
                         bool early, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(block, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- device helpers

// First statement of a kernel that launch_early may launch early (EARLY: the
// kernel is compiled for, and only ever given, an early launch; the plain
// variant carries none of this code, which measured 1-4 % slower on plain
// launches even with nothing to do).  In order: let the next kernel in the
// stream launch early too; ask the L2 for the first `pf_bytes` of this CTA's
// state head (threads 0..3 a quarter each; `head` 16-byte aligned, pf_bytes a
// multiple of 64, 0 for none); wait until the previous kernel has completed
// and its writes are visible.  Nothing is read or written before that wait:
// an L2 prefetch is a hint and changes no value a load returns, so the results
// are those of plain stream order whatever the previous kernel did.
template <bool EARLY>
__device__ __forceinline__ void early_start(const void *head, unsigned pf_bytes)
{
    if constexpr (EARLY) {
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        if (pf_bytes != 0 && threadIdx.x < 4) {
            const char *b = static_cast<const char *>(head) + threadIdx.x * (pf_bytes / 4);
            asm volatile("{ .reg .u64 ga; cvta.to.global.u64 ga, %0; cp.async.bulk.prefetch.L2.global [ga], %1; }"
                         :: "l"(b), "r"(pf_bytes / 4) : "memory");
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }
}

// Streaming 16-byte global load / store: the state is touched once per call,
// so keep it from displacing reusable lines (cache-streaming hint).
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ void st_stream16(void *p, uint4 v) {
    __stcs(reinterpret_cast<uint4 *>(p), v);
}
// Read-only 16-byte load through the non-coherent path (inputs shared by heads).
__device__ __forceinline__ float4 ld_ro_f4(const float *p) {
    return __ldg(reinterpret_cast<const float4 *>(p));
}

// Butterfly sum over groups of W consecutive lanes (W a power of two <= 32);
// every lane of the group ends with the group total.
template <int W>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int off = W / 2; off > 0; off >>= 1) x += __shfl_xor_sync(kFull, x, off);
    return x;
}

// The sums of NVAL values at once, each spread over the same W lanes (part[j] on every lane of the
// group: e.g. u and w of several rows, partial over the lanes' columns): a reduce-scatter with the
// butterfly's partners and order (offsets W/2 .. 1), so every sum is group_sum<W>'s bit for bit.
// While a lane carries more than one value, a level halves them: the lane keeps the half its partner
// gives away and adds the partner's copy; the remaining levels are plain butterfly steps.  NVAL - 1
// + log2(W / NVAL) shuffles instead of NVAL log2(W), in one chain of log2(W) levels.  Returns the sum
// this lane ends with: value (lane % W) / (W / NVAL), held by W / NVAL consecutive lanes.
template <int W, int NVAL>
__device__ __forceinline__ float reduce_scatter(float (&part)[NVAL], int lane) {
    static_assert(NVAL <= W && (NVAL & (NVAL - 1)) == 0 && (W & (W - 1)) == 0, "NVAL values over W lanes");
#pragma unroll
    for (int lvl = 0; (W >> (lvl + 1)) > 0; ++lvl) {
        const int off = W >> (lvl + 1), half = NVAL >> (lvl + 1);
        if (half > 0) {
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int j = 0; j < half; ++j) {
                const float keep = upper ? part[j + half] : part[j];
                const float send = upper ? part[j] : part[j + half];
                part[j] = keep + __shfl_xor_sync(kFull, send, off);
            }
        } else {
            part[0] += __shfl_xor_sync(kFull, part[0], off);
        }
    }
    return part[0];
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + __expf(-z)); }

__device__ __forceinline__ uint16_t bf16_bits_rn(float x) {
    __nv_bfloat16 b = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t *>(&b);
}

// One group of 32 values, one per lane of a warp, to int8 codes and a scale
// (logicaffeine_compile/codegen_cuda/gdn.rs, kernel `gdn_gate_norm_q`): scale =
// max |y| / 127 over the group (1 if all zero), code = y / scale rounded to the
// nearest integer, ties to even.  Both divisions are IEEE fp32 divisions.
__device__ __forceinline__ void quant_group32(float yv, int8_t *code, float *scale, int lane) {
    float am = fabsf(yv);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(kFull, am, off));
    const float sc = am > 0.f ? am / 127.0f : 1.0f;
    *code = (int8_t)__float2int_rn(yv / sc);
    if (lane == 0) *scale = sc;
}

// cp.async (global -> shared, bypassing L1) and its hardware group waits.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// A 16-byte vector of state elements, widened to / narrowed from fp32.
template <typename TS> struct Vec16;

template <> struct Vec16<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void unpack(const uint4 r, float (&x)[N]) {
        x[0] = __uint_as_float(r.x); x[1] = __uint_as_float(r.y);
        x[2] = __uint_as_float(r.z); x[3] = __uint_as_float(r.w);
    }
    __device__ __forceinline__ static uint4 pack(const float (&x)[N]) {
        return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]),
                          __float_as_uint(x[2]), __float_as_uint(x[3]));
    }
};

template <> struct Vec16<__half> {
    static constexpr int N = 8;
    __device__ __forceinline__ static float2 h2f(unsigned u) {
        __half2 h = *reinterpret_cast<__half2 *>(&u);
        return __half22float2(h);
    }
    __device__ __forceinline__ static unsigned f2h(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);           // round to nearest even
        return *reinterpret_cast<unsigned *>(&h);
    }
    __device__ __forceinline__ static void unpack(const uint4 r, float (&x)[N]) {
        float2 t;
        t = h2f(r.x); x[0] = t.x; x[1] = t.y;
        t = h2f(r.y); x[2] = t.x; x[3] = t.y;
        t = h2f(r.z); x[4] = t.x; x[5] = t.y;
        t = h2f(r.w); x[6] = t.x; x[7] = t.y;
    }
    __device__ __forceinline__ static uint4 pack(const float (&x)[N]) {
        return make_uint4(f2h(x[0], x[1]), f2h(x[2], x[3]), f2h(x[4], x[5]), f2h(x[6], x[7]));
    }
};

template <typename TS> __device__ __forceinline__ float to_f32(TS x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <typename TS> __device__ __forceinline__ TS from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }

}  // namespace gdn
