// gdn_abi.cu -- the extern "C" entry points of libgdn (declared in
// include/gdn.h): argument checks on the host, then one kernel launch.
//
// Every check runs before any CUDA call, so a rejected call has no effect and
// the checks can be exercised on a machine without a GPU.
#include <cmath>
#include <cstdint>

#include "gdn.h"
#include "gdn_internal.cuh"
#include "gdn_tc.cuh"

namespace gdn {

int sm_count()
{
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

namespace {

thread_local int t_last_cuda_error = 0;

int cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return GDN_OK;
    t_last_cuda_error = (int)e;
    return GDN_ERR_CUDA;
}

// A byte range [lo, hi) touched by one operand.
struct Span {
    uintptr_t lo, hi;
};

// Bytes spanned by `rows` rows of `len` elements, `stride` elements apart.
bool rows_span(const void *base, int64_t rows, int64_t len, int64_t stride, int64_t elem, Span *out)
{
    if (rows <= 0 || len <= 0) { out->lo = out->hi = (uintptr_t)base; return true; }
    // (rows - 1) * stride + len elements, guarding 64-bit overflow
    if (stride > 0 && rows - 1 > (INT64_MAX - len) / stride) return false;
    const int64_t elems = (rows - 1) * stride + len;
    if (elems > INT64_MAX / elem) return false;
    out->lo = (uintptr_t)base;
    out->hi = out->lo + (uintptr_t)(elems * elem);
    return out->hi >= out->lo;
}

bool overlap(const Span &a, const Span &b) { return a.lo < b.hi && b.lo < a.hi; }

bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

// Checks shared by decode and prefill.  `rows` is the number of token rows
// (batch for decode, batch * seq_len for prefill).
struct Operand {
    const void *p;
    int64_t rows, len, stride, elem;
};

int check_common(int batch, int nk, int nv, int d, int64_t pitch, int state_dtype)
{
    if (batch < 0 || nk <= 0 || nv <= 0 || d <= 0) return GDN_ERR_ARG;
    if (state_dtype != GDN_STATE_F32 && state_dtype != GDN_STATE_F16) return GDN_ERR_UNSUPPORTED;
    if (d > 256) return GDN_ERR_UNSUPPORTED;
    if ((int64_t)batch * nv > INT32_MAX) return GDN_ERR_UNSUPPORTED;
    const int64_t head_elems = (int64_t)nv * d * d;
    if (pitch < head_elems) return GDN_ERR_ARG;
    return GDN_OK;
}

// Every operand: non-null, stride >= row length, element-aligned; outputs
// (the first `n_out` entries) overlap nothing else.
int check_operands(const Operand *ops, int n_ops, int n_out)
{
    Span spans[16];
    for (int i = 0; i < n_ops; ++i) {
        const Operand &o = ops[i];
        if (o.p == nullptr) return GDN_ERR_ARG;
        if (o.rows > 1 && o.stride < o.len) return GDN_ERR_ARG;
        if (!aligned(o.p, (uintptr_t)o.elem)) return GDN_ERR_ALIGN;
        if (!rows_span(o.p, o.rows, o.len, o.stride, o.elem, &spans[i])) return GDN_ERR_ARG;
    }
    for (int i = 0; i < n_out; ++i)
        for (int j = 0; j < n_ops; ++j)
            if (j != i && overlap(spans[i], spans[j])) return GDN_ERR_ALIAS;
    return GDN_OK;
}

bool vec16(const void *p) { return aligned(p, 16); }

float inv_sqrt(int d) { return (float)(1.0 / std::sqrt((double)d)); }

// What a single-token call writes besides the state: raw fp32 o, the normed
// output as bf16, or the normed output as int8 groups of 32 (plus, optionally,
// the fp32 normed values).
struct Epilogue {
    int kind;                                   // kEpiRaw, kEpiBf16, kEpiQ8
    float *o = nullptr;          int64_t o_stride = 0;
    uint16_t *out = nullptr;     int64_t out_stride = 0;
    int8_t *xq = nullptr;        int64_t xq_stride = 0;
    float *xs = nullptr;         int64_t xs_stride = 0;
    float *y = nullptr;          int64_t y_stride = 0;
};

int decode_entry(void *state, int state_dtype, int64_t state_pitch,
                 const float *q, const float *k, const float *v,
                 const float *alpha, const float *beta,
                 const float *z, const float *gn, float eps,
                 const Epilogue &ep,
                 int batch, int nk, int nv, int d,
                 int64_t qk_stride, int64_t v_stride, int64_t gb_stride,
                 int64_t z_stride, void *stream)
{
    int st = check_common(batch, nk, nv, d, state_pitch, state_dtype);
    if (st != GDN_OK) return st;
    const bool norm = ep.kind != kEpiRaw;
    if (norm && !(eps >= 0.0f && std::isfinite(eps))) return GDN_ERR_ARG;
    if (ep.kind == kEpiQ8 && d % 32 != 0) return GDN_ERR_UNSUPPORTED;   // groups of 32 inside a head
    const int64_t selem = state_dtype == GDN_STATE_F16 ? 2 : 4;
    const int64_t B = batch, hv = (int64_t)nv * d, hk = (int64_t)nk * d;
    Operand ops[12];
    int n = 0;
    ops[n++] = {state, B, (int64_t)nv * d * d, state_pitch, selem};
    if (ep.kind == kEpiBf16) {
        ops[n++] = {ep.out, B, hv, ep.out_stride, 2};
    } else if (ep.kind == kEpiQ8) {
        ops[n++] = {ep.xq, B, hv, ep.xq_stride, 1};
        ops[n++] = {ep.xs, B, hv / 32, ep.xs_stride, 4};
        if (ep.y != nullptr) ops[n++] = {ep.y, B, hv, ep.y_stride, 4};
    } else {
        ops[n++] = {ep.o, B, hv, ep.o_stride, 4};
    }
    const int n_out = n;
    ops[n++] = {q, B, hk, qk_stride, 4};
    ops[n++] = {k, B, hk, qk_stride, 4};
    ops[n++] = {v, B, hv, v_stride, 4};
    ops[n++] = {alpha, B, nv, gb_stride, 4};
    ops[n++] = {beta, B, nv, gb_stride, 4};
    if (norm) {
        ops[n++] = {z, B, hv, z_stride, 4};
        ops[n++] = {gn, 1, d, d, 4};
    }
    if (batch == 0) {
        // empty call: still reject null pointers, nothing to launch
        for (int i = 0; i < n; ++i) if (ops[i].p == nullptr) return GDN_ERR_ARG;
        return GDN_OK;
    }
    st = check_operands(ops, n, n_out);
    if (st != GDN_OK) return st;

    DecodeParams p{};
    p.state = state; p.pitch = state_pitch;
    p.q = q; p.k = k; p.v = v; p.alpha = alpha; p.beta = beta;
    p.z = z; p.gn = gn; p.o = ep.o; p.out = ep.out;
    p.xq = ep.xq; p.xs = ep.xs; p.y = ep.y;
    p.qk_stride = qk_stride; p.v_stride = v_stride; p.gb_stride = gb_stride;
    p.z_stride = z_stride; p.o_stride = ep.o_stride; p.out_stride = ep.out_stride;
    p.xq_stride = ep.xq_stride; p.xs_stride = ep.xs_stride; p.y_stride = ep.y_stride;
    p.batch = batch; p.nk = nk; p.nv = nv; p.d = d;
    p.eps = eps; p.inv_sqrt_d = inv_sqrt(d);

    // D == 128 vector path: 16-byte state rows and 16-byte k/q columns.
    // (v, z, gn, alpha, beta, o and out are read/written as scalars.)
    const bool fast = d == 128 && vec16(state) && (state_pitch * selem) % 16 == 0 &&
                      vec16(q) && vec16(k) && (qk_stride * 4) % 16 == 0;
    return cuda_status(launch_decode(p, state_dtype == GDN_STATE_F16, ep.kind, fast, (cudaStream_t)stream));
}

}  // namespace

int report_cuda_error(cudaError_t e) { return cuda_status(e); }

// gdn_decode_conv_norm's checks and launch.  With `counters_of` set (the
// allocation-free entry) the workspace argument is ignored and the counters'
// device address comes from counters_of, called only after every argument has
// passed its checks, so a rejected or empty call makes no CUDA call at all.
int decode_conv_norm_entry(void *state, int state_dtype, int64_t state_pitch,
                           float *conv_state, int64_t conv_pitch, int taps,
                           const float *x, const float *conv_w,
                           const float *br, const float *ar, const float *dt, const float *rate,
                           const float *z, const float *gn, float l2_eps, float eps,
                           uint16_t *out, int32_t *workspace, CountersFn counters_of,
                           int batch, int nk, int nv, int d,
                           int64_t x_stride, int64_t gate_stride, int64_t z_stride,
                           int64_t out_stride, void *stream)
{
    int st = check_common(batch, nk, nv, d, state_pitch, state_dtype);
    if (st != GDN_OK) return st;
    if (nv % nk != 0) return GDN_ERR_UNSUPPORTED;
    if (taps < 1 || taps > 8) return GDN_ERR_ARG;
    if (!(eps >= 0.0f && std::isfinite(eps)) || !(l2_eps >= 0.0f && std::isfinite(l2_eps))) return GDN_ERR_ARG;
    const int repeat = nv / nk;
    // the general kernel keeps q, k, every value head's v, o and the gates in shared memory
    if ((size_t)(3 + repeat) * d * 4 + 8 * (size_t)repeat > 48 * 1024) return GDN_ERR_UNSUPPORTED;
    const int64_t selem = state_dtype == GDN_STATE_F16 ? 2 : 4;
    const int64_t B = batch, hv = (int64_t)nv * d, C = (int64_t)(2 * nk + nv) * d;
    if (conv_pitch < taps * C) return GDN_ERR_ARG;
    Operand ops[12] = {
        {state, B, (int64_t)nv * d * d, state_pitch, selem},
        {conv_state, B, taps * C, conv_pitch, 4},
        {out, B, hv, out_stride, 2},
        {workspace, 1, B * nk, B * nk, 4},
        {x, B, C, x_stride, 4},
        {conv_w, 1, taps * C, taps * C, 4},
        {br, B, nv, gate_stride, 4},
        {ar, B, nv, gate_stride, 4},
        {dt, 1, nv, nv, 4},
        {rate, 1, nv, nv, 4},
        {z, B, hv, z_stride, 4},
        {gn, 1, d, d, 4},
    };
    // with counters_of set, the counters are the library's own, not an operand of the call
    const int n_ops = counters_of ? 11 : 12;
    if (counters_of) ops[3] = ops[11];
    if (batch == 0) {
        for (int i = 0; i < n_ops; ++i) if (ops[i].p == nullptr) return GDN_ERR_ARG;
        return GDN_OK;
    }
    st = check_operands(ops, n_ops, counters_of ? 3 : 4);
    if (st != GDN_OK) return st;
    if (counters_of) {                       // every check has passed: now the CUDA call
        const cudaError_t e = counters_of(&workspace);
        if (e != cudaSuccess) return cuda_status(e);
    }

    ConvNormParams p{};
    p.state = state; p.pitch = state_pitch;
    p.ring = conv_state; p.ring_pitch = conv_pitch;
    p.x = x; p.x_stride = x_stride; p.w = conv_w;
    p.br = br; p.ar = ar; p.gate_stride = gate_stride; p.dt = dt; p.rate = rate;
    p.z = z; p.gn = gn; p.out = out; p.z_stride = z_stride; p.out_stride = out_stride;
    p.counters = workspace;
    p.batch = batch; p.nk = nk; p.nv = nv; p.d = d; p.taps = taps; p.repeat = repeat;
    p.l2_eps = l2_eps; p.eps = eps; p.inv_sqrt_d = inv_sqrt(d);
    // D == 128 kernel: 16-byte state rows
    const bool fast = d == 128 && vec16(state) && (state_pitch * selem) % 16 == 0;
    return cuda_status(launch_conv_norm(p, state_dtype == GDN_STATE_F16, fast, (cudaStream_t)stream));
}


namespace {

// The standalone gated norm: rows of NV heads x D raw outputs o (and gate
// inputs z) to the bf16 or int8 epilogue.  Checks as for decode.
int norm_entry(const float *o, const float *z, const float *gn, float eps, NormParams p, int epi,
               int64_t rows, int nv, int d, int64_t o_stride, int64_t z_stride, void *stream)
{
    if (rows < 0 || nv <= 0 || d <= 0) return GDN_ERR_ARG;
    if (d > 256) return GDN_ERR_UNSUPPORTED;
    if (epi == kEpiQ8 && d % 32 != 0) return GDN_ERR_UNSUPPORTED;
    if (!(eps >= 0.0f && std::isfinite(eps))) return GDN_ERR_ARG;
    if (rows > INT64_MAX / nv || rows * nv > (int64_t)INT32_MAX * 8) return GDN_ERR_UNSUPPORTED;   // grid size
    const int64_t hv = (int64_t)nv * d;
    Operand ops[7];
    int n = 0;
    if (epi == kEpiBf16) {
        ops[n++] = {p.out, rows, hv, p.out_stride, 2};
    } else {
        ops[n++] = {p.xq, rows, hv, p.xq_stride, 1};
        ops[n++] = {p.xs, rows, hv / 32, p.xs_stride, 4};
        if (p.y != nullptr) ops[n++] = {p.y, rows, hv, p.y_stride, 4};
    }
    const int n_out = n;
    ops[n++] = {o, rows, hv, o_stride, 4};
    ops[n++] = {z, rows, hv, z_stride, 4};
    ops[n++] = {gn, 1, d, d, 4};
    if (rows == 0) {
        for (int i = 0; i < n; ++i) if (ops[i].p == nullptr) return GDN_ERR_ARG;
        return GDN_OK;
    }
    const int st = check_operands(ops, n, n_out);
    if (st != GDN_OK) return st;
    p.o = o; p.z = z; p.gn = gn; p.eps = eps;
    p.rows = rows; p.nv = nv; p.d = d; p.o_stride = o_stride; p.z_stride = z_stride;
    // D == 128 vector kernel: 16-byte o, z, gn rows; 8-byte bf16 or 4-byte int8 and 16-byte y rows
    bool fast = d == 128 && vec16(o) && vec16(z) && vec16(gn) && (o_stride * 4) % 16 == 0 &&
                (z_stride * 4) % 16 == 0;
    if (epi == kEpiBf16) {
        fast = fast && aligned(p.out, 8) && (p.out_stride * 2) % 8 == 0;
    } else {
        fast = fast && aligned(p.xq, 4) && p.xq_stride % 4 == 0 &&
               (p.y == nullptr || (vec16(p.y) && (p.y_stride * 4) % 16 == 0));
    }
    return cuda_status(launch_gate_norm(p, epi, fast, (cudaStream_t)stream));
}

}  // namespace

// gdn_prefill_seq and gdn_prefill_chunked: the same checks; `chunked` takes the
// tensor-core kernel where it applies (D == 128, 16-byte k and q rows).
int prefill_entry(void *state, int state_dtype, int64_t state_pitch,
                  const float *q, const float *k, const float *v,
                  const float *alpha, const float *beta, float *o,
                  int batch, int seq_len, int nk, int nv, int d,
                  int64_t qk_stride, int64_t v_stride, int64_t gb_stride,
                  int64_t o_stride, void *stream, bool chunked)
{
    int st = check_common(batch, nk, nv, d, state_pitch, state_dtype);
    if (st != GDN_OK) return st;
    if (seq_len < 0) return GDN_ERR_ARG;
    const int64_t selem = state_dtype == GDN_STATE_F16 ? 2 : 4;
    const int64_t B = batch, R = (int64_t)batch * seq_len;
    const int64_t hv = (int64_t)nv * d, hk = (int64_t)nk * d;
    Operand ops[7] = {
        {state, B, (int64_t)nv * d * d, state_pitch, selem},
        {o, R, hv, o_stride, 4},
        {q, R, hk, qk_stride, 4},
        {k, R, hk, qk_stride, 4},
        {v, R, hv, v_stride, 4},
        {alpha, R, nv, gb_stride, 4},
        {beta, R, nv, gb_stride, 4},
    };
    if (R == 0) {
        for (auto &op : ops) if (op.p == nullptr) return GDN_ERR_ARG;
        return GDN_OK;
    }
    st = check_operands(ops, 7, 2);
    if (st != GDN_OK) return st;

    PrefillParams p{};
    p.state = state; p.pitch = state_pitch;
    p.q = q; p.k = k; p.v = v; p.alpha = alpha; p.beta = beta; p.o = o;
    p.qk_stride = qk_stride; p.v_stride = v_stride; p.gb_stride = gb_stride; p.o_stride = o_stride;
    p.batch = batch; p.seq_len = seq_len; p.nk = nk; p.nv = nv; p.d = d;
    p.inv_sqrt_d = inv_sqrt(d);
    p.zero = 0;
    // D == 128 path: 16-byte state rows, 16-byte k/q rows and 16-byte v row blocks
    const bool fast = d == 128 && vec16(state) && (state_pitch * selem) % 16 == 0 &&
                      vec16(q) && vec16(k) && (qk_stride * 4) % 16 == 0 &&
                      vec16(v) && (v_stride * 4) % 16 == 0;
    if (chunked && d == 128 && vec16(q) && vec16(k) && (qk_stride * 4) % 16 == 0)
        return cuda_status(launch_prefill_tc(p, state_dtype == GDN_STATE_F16, (cudaStream_t)stream));
    return cuda_status(launch_prefill(p, state_dtype == GDN_STATE_F16, fast, (cudaStream_t)stream));
}


}  // namespace gdn

using namespace gdn;

extern "C" {

GDN_API int gdn_decode(void *state, gdn_state_dtype state_dtype, int64_t state_pitch,
                       const float *q, const float *k, const float *v,
                       const float *alpha, const float *beta, float *o,
                       int batch, int nk, int nv, int d,
                       int64_t qk_stride, int64_t v_stride, int64_t gb_stride,
                       int64_t o_stride, void *stream)
{
    Epilogue ep{kEpiRaw};
    ep.o = o; ep.o_stride = o_stride;
    return decode_entry(state, state_dtype, state_pitch, q, k, v, alpha, beta, nullptr, nullptr, 0.0f,
                        ep, batch, nk, nv, d, qk_stride, v_stride, gb_stride, 0, stream);
}

GDN_API int gdn_decode_norm(void *state, gdn_state_dtype state_dtype, int64_t state_pitch,
                            const float *q, const float *k, const float *v,
                            const float *alpha, const float *beta,
                            const float *z, const float *gn, float eps,
                            uint16_t *out,
                            int batch, int nk, int nv, int d,
                            int64_t qk_stride, int64_t v_stride, int64_t gb_stride,
                            int64_t z_stride, int64_t out_stride, void *stream)
{
    Epilogue ep{kEpiBf16};
    ep.out = out; ep.out_stride = out_stride;
    return decode_entry(state, state_dtype, state_pitch, q, k, v, alpha, beta, z, gn, eps,
                        ep, batch, nk, nv, d, qk_stride, v_stride, gb_stride, z_stride, stream);
}

GDN_API int gdn_decode_norm_q8(void *state, gdn_state_dtype state_dtype, int64_t state_pitch,
                               const float *q, const float *k, const float *v,
                               const float *alpha, const float *beta,
                               const float *z, const float *gn, float eps,
                               int8_t *xq, float *xs, float *y,
                               int batch, int nk, int nv, int d,
                               int64_t qk_stride, int64_t v_stride, int64_t gb_stride,
                               int64_t z_stride, int64_t xq_stride, int64_t xs_stride,
                               int64_t y_stride, void *stream)
{
    Epilogue ep{kEpiQ8};
    ep.xq = xq; ep.xq_stride = xq_stride;
    ep.xs = xs; ep.xs_stride = xs_stride;
    ep.y = y; ep.y_stride = y_stride;
    return decode_entry(state, state_dtype, state_pitch, q, k, v, alpha, beta, z, gn, eps,
                        ep, batch, nk, nv, d, qk_stride, v_stride, gb_stride, z_stride, stream);
}

GDN_API int gdn_decode_conv_norm(void *state, gdn_state_dtype state_dtype, int64_t state_pitch,
                                 float *conv_state, int64_t conv_pitch, int taps,
                                 const float *x, const float *conv_w,
                                 const float *br, const float *ar, const float *dt, const float *rate,
                                 const float *z, const float *gn, float l2_eps, float eps,
                                 uint16_t *out, int32_t *workspace,
                                 int batch, int nk, int nv, int d,
                                 int64_t x_stride, int64_t gate_stride, int64_t z_stride,
                                 int64_t out_stride, void *stream)
{
    return gdn::decode_conv_norm_entry(state, state_dtype, state_pitch, conv_state, conv_pitch, taps, x, conv_w,
                                       br, ar, dt, rate, z, gn, l2_eps, eps, out, workspace, nullptr,
                                       batch, nk, nv, d, x_stride, gate_stride, z_stride, out_stride, stream);
}

GDN_API int gdn_decode_chunk2(void *state, gdn_state_dtype state_dtype, int64_t state_pitch,
                              void *state_mid, int64_t mid_pitch,
                              const float *q, const float *k, const float *v,
                              const float *alpha, const float *beta, float *o,
                              int batch, int nk, int nv, int d,
                              int64_t qk_stride, int64_t v_stride, int64_t gb_stride,
                              int64_t o_stride, void *stream)
{
    int st = check_common(batch, nk, nv, d, state_pitch, state_dtype);
    if (st != GDN_OK) return st;
    if (mid_pitch < (int64_t)nv * d * d) return GDN_ERR_ARG;
    const int64_t selem = state_dtype == GDN_STATE_F16 ? 2 : 4;
    const int64_t B = batch, R = 2 * (int64_t)batch;
    const int64_t hv = (int64_t)nv * d, hk = (int64_t)nk * d;
    Operand ops[8] = {
        {state, B, (int64_t)nv * d * d, state_pitch, selem},
        {state_mid, B, (int64_t)nv * d * d, mid_pitch, selem},
        {o, R, hv, o_stride, 4},
        {q, R, hk, qk_stride, 4},
        {k, R, hk, qk_stride, 4},
        {v, R, hv, v_stride, 4},
        {alpha, R, nv, gb_stride, 4},
        {beta, R, nv, gb_stride, 4},
    };
    if (batch == 0) {
        for (auto &op : ops) if (op.p == nullptr) return GDN_ERR_ARG;
        return GDN_OK;
    }
    st = check_operands(ops, 8, 3);
    if (st != GDN_OK) return st;

    DecodeParams p{};
    p.state = state; p.pitch = state_pitch;
    p.state_mid = state_mid; p.mid_pitch = mid_pitch;
    p.q = q; p.k = k; p.v = v; p.alpha = alpha; p.beta = beta; p.o = o;
    p.qk_stride = qk_stride; p.v_stride = v_stride; p.gb_stride = gb_stride; p.o_stride = o_stride;
    p.batch = batch; p.nk = nk; p.nv = nv; p.d = d;
    p.inv_sqrt_d = inv_sqrt(d);
    const bool fast = d == 128 && vec16(state) && (state_pitch * selem) % 16 == 0 &&
                      vec16(state_mid) && (mid_pitch * selem) % 16 == 0 &&
                      vec16(q) && vec16(k) && (qk_stride * 4) % 16 == 0;
    return cuda_status(launch_decode_chunk2(p, state_dtype == GDN_STATE_F16, fast, (cudaStream_t)stream));
}

GDN_API int gdn_prefill_seq(void *state, gdn_state_dtype state_dtype, int64_t state_pitch,
                            const float *q, const float *k, const float *v,
                            const float *alpha, const float *beta, float *o,
                            int batch, int seq_len, int nk, int nv, int d,
                            int64_t qk_stride, int64_t v_stride, int64_t gb_stride,
                            int64_t o_stride, void *stream)
{
    return prefill_entry(state, state_dtype, state_pitch, q, k, v, alpha, beta, o, batch, seq_len, nk, nv, d,
                         qk_stride, v_stride, gb_stride, o_stride, stream, false);
}

GDN_API int gdn_prefill_chunked(void *state, gdn_state_dtype state_dtype, int64_t state_pitch,
                                const float *q, const float *k, const float *v,
                                const float *alpha, const float *beta, float *o,
                                int batch, int seq_len, int nk, int nv, int d,
                                int64_t qk_stride, int64_t v_stride, int64_t gb_stride,
                                int64_t o_stride, void *stream)
{
    return prefill_entry(state, state_dtype, state_pitch, q, k, v, alpha, beta, o, batch, seq_len, nk, nv, d,
                         qk_stride, v_stride, gb_stride, o_stride, stream, true);
}

GDN_API int gdn_device_wait_timeouts(unsigned *count)
{
    if (count == nullptr) return GDN_ERR_ARG;
    return cuda_status(tc_wait_timeouts(count));
}

GDN_API void gdn_set_wait_polls(unsigned polls) { tc_set_wait_polls(polls); }

GDN_API void gdn_set_mma_wait_polls(unsigned polls) { tc_set_mma_wait_polls(polls); }

GDN_API int gdn_gate_norm(const float *o, const float *z, const float *gn, float eps, uint16_t *out,
                          int64_t rows, int nv, int d, int64_t o_stride, int64_t z_stride,
                          int64_t out_stride, void *stream)
{
    NormParams p{};
    p.out = out; p.out_stride = out_stride;
    return norm_entry(o, z, gn, eps, p, kEpiBf16, rows, nv, d, o_stride, z_stride, stream);
}

GDN_API int gdn_gate_norm_q8(const float *o, const float *z, const float *gn, float eps,
                             int8_t *xq, float *xs, float *y, int64_t rows, int nv, int d,
                             int64_t o_stride, int64_t z_stride, int64_t xq_stride, int64_t xs_stride,
                             int64_t y_stride, void *stream)
{
    NormParams p{};
    p.xq = xq; p.xq_stride = xq_stride;
    p.xs = xs; p.xs_stride = xs_stride;
    p.y = y; p.y_stride = y_stride;
    return norm_entry(o, z, gn, eps, p, kEpiQ8, rows, nv, d, o_stride, z_stride, stream);
}

GDN_API int gdn_h_f32_to_f16(const float *src, uint16_t *dst, uint64_t n, void *stream)
{
    if (src == nullptr || dst == nullptr) return GDN_ERR_ARG;
    if (n == 0) return GDN_OK;
    if (n > (uint64_t)INT64_MAX / 4) return GDN_ERR_ARG;
    if (!aligned(src, 4) || !aligned(dst, 2)) return GDN_ERR_ALIGN;
    const Span a{(uintptr_t)src, (uintptr_t)src + n * 4}, b{(uintptr_t)dst, (uintptr_t)dst + n * 2};
    if (overlap(a, b)) return GDN_ERR_ALIAS;
    return cuda_status(launch_f32_to_f16(src, dst, n, vec16(src) && vec16(dst), (cudaStream_t)stream));
}

GDN_API int gdn_h_f16_to_f32(const uint16_t *src, float *dst, uint64_t n, void *stream)
{
    if (src == nullptr || dst == nullptr) return GDN_ERR_ARG;
    if (n == 0) return GDN_OK;
    if (n > (uint64_t)INT64_MAX / 4) return GDN_ERR_ARG;
    if (!aligned(src, 2) || !aligned(dst, 4)) return GDN_ERR_ALIGN;
    const Span a{(uintptr_t)src, (uintptr_t)src + n * 2}, b{(uintptr_t)dst, (uintptr_t)dst + n * 4};
    if (overlap(a, b)) return GDN_ERR_ALIAS;
    return cuda_status(launch_f16_to_f32(src, dst, n, vec16(src) && vec16(dst), (cudaStream_t)stream));
}

GDN_API const char *gdn_status_str(int status)
{
    switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_ARG: return "GDN_ERR_ARG: invalid argument (null pointer, bad size, short stride or pitch, bad eps)";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: unsupported shape or state dtype";
    case GDN_ERR_ALIGN: return "GDN_ERR_ALIGN: pointer not aligned to its element size";
    case GDN_ERR_ALIAS: return "GDN_ERR_ALIAS: an output overlaps another operand";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA: CUDA launch failed";
    default: return "GDN_ERR_UNKNOWN";
    }
}

GDN_API int gdn_last_cuda_error(void) { return t_last_cuda_error; }

}  // extern "C"
