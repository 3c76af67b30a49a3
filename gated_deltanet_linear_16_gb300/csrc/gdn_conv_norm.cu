// gdn_conv_norm.cu -- one decode token from the projection outputs to the
// normed bf16 output in a single launch: the depthwise causal conv ring update
// with silu on q, k and v, the per-head L2 normalisation of q and k, the two
// gates from their logits, the gated delta rule step and the gated RMS norm.
//
// Follows metrale_model_layers/layers/ops/ssm_gdn_a.rs, launcher
// `gdn_decode_f32_conv_norm` (conv update, L2 norm, recurrence and gated norm
// in one decode launch; each ring row has exactly one writer), and
// logicaffeine_compile/codegen_cuda/gdn.rs: `gk_conv_silu_l2` (shift the ring
// by one, append the token, reduce with the taps, silu; L2 of the q/k heads
// with den = sqrt(sum x^2 + eps)), `gk_gdn_gates` (beta = sigmoid(br), alpha
// = (1 + e^(ar + dt))^rate with rate the stored negative decay rate),
// `gdn_step` and `gdn_gate_norm`.
//
// GB300 design.  The page's launcher gives one block to a key head and its
// NV/NK value heads.  For fp32 states every value head keeps one CTA here --
// the decode kernel's shape (8 warps x 16 rows), so the 64 KB-per-head state
// stream is unchanged and no CTA waits for another (fp16 states take the
// page's per-key-head shape, conv_norm_kh below, which measured faster there):
//  * every CTA issues its conv inputs first (ring entries, token values, tap
//    weights: a few KB that would otherwise queue behind the state stream),
//    then its state loads, then computes while the state streams in;
//  * it updates the ring rows of its own value head's v channels and computes
//    v (one writer per ring row);
//  * it also computes the key head's q and k (conv, silu, L2: 256 channels)
//    from the ring as it was, without writing it, and keeps the shifted rows in
//    shared memory;
//  * after reading, a CTA counts itself in a per-(sequence, key head) counter
//    (fence + atomic add by one thread as its last batch of rows begins, the
//    result read only after the step); the CTA that completes the count is the
//    last reader of those ring rows, so it writes them and resets the counter.
// No barrier spans CTAs and nothing spins.  (Thread-block clusters, tried
// first for this exchange, cost ~30 % on GB300: co-scheduling the cluster's
// CTAs left SM slots idle.)
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kD = 128;
constexpr int kWarps = 8;
constexpr int kRowsPerWarp = kD / kWarps;   // 16

constexpr int kMaxTaps = 8;                 // the host rejects more

// One channel's stored inputs: the taps - 1 ring entries that stay in the ring
// (oldest first) and the token's value; MT bounds the tap count (the arrays
// live in registers, so a call with few taps takes an instance with a small
// MT).  Callers load every channel they own first, then compute, then store
// the shifted rows: a store through a generic pointer between two loads would
// keep the later load behind it, costing a second memory latency.
template <int MT>
struct ConvIn {
    float val[MT - 1];
    float xv;
};

template <int MT>
__device__ __forceinline__ void conv_load(ConvIn<MT> &in, const float *ring, const float *x, int64_t c, int64_t C,
                                          int taps) {
#pragma unroll
    for (int t = 0; t + 1 < MT; ++t) in.val[t] = t + 1 < taps ? ring[(int64_t)(t + 1) * C + c] : 0.f;
    in.xv = __ldg(x + c);
}

// The conv over the shifted ring (taps in order, the new token last) and silu.
template <int MT>
__device__ __forceinline__ float conv_silu(const ConvIn<MT> &in, const float *w, int64_t c, int64_t C, int taps) {
    float acc = 0.f;
#pragma unroll
    for (int t = 0; t + 1 < MT; ++t)
        if (t + 1 < taps) acc = fmaf(in.val[t], __ldg(w + (int64_t)t * C + c), acc);
    acc = fmaf(in.xv, __ldg(w + (int64_t)(taps - 1) * C + c), acc);
    return silu(acc);
}

// The ring's new contents (shift up by one, append the token) to `dst` (taps
// entries, stride `stride`): the ring itself for the channel's only writer, or
// a shared-memory copy for a later writer.
template <int MT>
__device__ __forceinline__ void conv_shift(const ConvIn<MT> &in, float *dst, int64_t stride, int taps) {
#pragma unroll
    for (int t = 0; t + 1 < MT; ++t)
        if (t + 1 < taps) dst[(int64_t)t * stride] = in.val[t];
    dst[(int64_t)(taps - 1) * stride] = in.xv;
}

// A channel's stored inputs with its taps' weights, all loaded at once (the
// per-value-head kernel issues these before its state stream, which would
// otherwise queue ahead of them).
template <int MT>
struct ConvInW {
    ConvIn<MT> in;
    float wt[MT - 1];
    float wx;
};

template <int MT>
__device__ __forceinline__ void conv_load_w(ConvInW<MT> &c, const float *ring, const float *x, const float *w,
                                            int64_t ch, int64_t C, int taps) {
    conv_load(c.in, ring, x, ch, C, taps);
#pragma unroll
    for (int t = 0; t + 1 < MT; ++t) c.wt[t] = t + 1 < taps ? __ldg(w + (int64_t)t * C + ch) : 0.f;
    c.wx = __ldg(w + (int64_t)(taps - 1) * C + ch);
}

// conv_silu over preloaded weights (the same arithmetic in the same order).
template <int MT>
__device__ __forceinline__ float conv_silu_w(const ConvInW<MT> &c, int taps) {
    float acc = 0.f;
#pragma unroll
    for (int t = 0; t + 1 < MT; ++t)
        if (t + 1 < taps) acc = fmaf(c.in.val[t], c.wt[t], acc);
    acc = fmaf(c.in.xv, c.wx, acc);
    return silu(acc);
}

// One channel through the conv ring in place: shift, append, reduce, silu.
// The caller is the only thread touching this channel.
__device__ __forceinline__ float conv_silu_channel(float *ring, const float *x, const float *w,
                                                   int64_t c, int64_t C, int taps) {
    ConvIn<kMaxTaps> in;
    conv_load(in, ring, x, c, C, taps);
    const float y = conv_silu(in, w, c, C, taps);
    conv_shift(in, ring + c, C, taps);
    return y;
}

__device__ __forceinline__ void gates(const ConvNormParams &p, int seq, int h, float &alpha, float &beta) {
    const float br = __ldg(p.br + seq * p.gate_stride + h);
    const float ar = __ldg(p.ar + seq * p.gate_stride + h);
    beta = 1.0f / (1.0f + expf(-br));
    alpha = powf(1.0f + expf(ar + __ldg(p.dt + h)), __ldg(p.rate + h));
}

// The gates' four inputs, loaded apart from their arithmetic (gates_of) so the
// loads can be in flight with a thread's other producer loads.
struct GateIn { float br, ar, dt, rate; };
__device__ __forceinline__ GateIn gate_load(const ConvNormParams &p, int seq, int h) {
    return {__ldg(p.br + seq * p.gate_stride + h), __ldg(p.ar + seq * p.gate_stride + h), __ldg(p.dt + h),
            __ldg(p.rate + h)};
}
__device__ __forceinline__ void gates_of(const GateIn &g, float &alpha, float &beta) {
    beta = 1.0f / (1.0f + expf(-g.br));
    alpha = powf(1.0f + expf(g.ar + g.dt), g.rate);
}

constexpr int kGroups = 4;                 // cp.async commit groups per lane (staged)

template <typename TS>
constexpr int stage_bytes() { return kD * kD * (int)sizeof(TS); }

// STAGED: the head's state goes to shared memory by cp.async, every load in
// flight at once (as the staged decode kernel); otherwise NB register batches.
template <typename TS, bool STAGED, int NB, int MINB, bool EARLY, int MT>
__global__ void __launch_bounds__(kWarps * 32, MINB)
conv_norm_d128(const ConvNormParams p)
{
    using V = Vec16<TS>;
    constexpr int EPV = V::N;
    constexpr int LPR = kD / EPV;
    constexpr int RPL = 32 / LPR;
    constexpr int NLD = kRowsPerWarp / RPL;
    constexpr int VPR = kD * (int)sizeof(TS) / 16;
    constexpr int NBAT = STAGED ? kGroups : NB;
    constexpr int PER = NLD / NBAT;
    static_assert(NLD % NBAT == 0, "shape");

    __shared__ __align__(16) float q_s[kD];
    __shared__ __align__(16) float k_s[kD];
    __shared__ float v_s[kD];
    __shared__ float red_q[4], red_k[4], red[kWarps];
    __shared__ float gate_s[2];
    __shared__ float ring_new[2][8][kD];                 // the key head's new q/k ring rows
    __shared__ int last_reader;

    const int cl = blockIdx.x / p.repeat;               // (sequence, key head)
    const int rank = blockIdx.x - cl * p.repeat;        // which value head of the key head
    const int seq = cl / p.nk;
    const int kh = cl - seq * p.nk;
    const int h = kh + (int)rank * p.nk;                // tiled pairing: h mod NK == kh
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sub = lane / LPR;
    const int col = (lane % LPR) * EPV;
    const int row0 = warp * kRowsPerWarp;
    const int64_t C = (int64_t)(2 * p.nk + p.nv) * kD;

    TS *head = reinterpret_cast<TS *>(p.state) + seq * p.pitch + (int64_t)h * kD * kD;
    TS *rowp = head + (int64_t)(row0 + sub) * kD + col;
    early_start<EARLY>(head, p.pf_bytes);

    // 1. the producers' inputs: a few KB per CTA, issued before the state stream so that they do not
    //    queue behind it.  Threads 0..127: channel i of this value head's v (ring rows written below,
    //    by their only writer) and thread 0 the gate inputs; threads 128..255: channel i of the key
    //    head's q and of its k (read only; the last reader writes them, step 6).
    float *ring = p.ring + seq * p.ring_pitch;
    const float *x = p.x + seq * p.x_stride;
    const int pi = tid & (kD - 1);
    const int64_t cv = 2 * (int64_t)p.nk * kD + (int64_t)h * kD + pi;
    const int64_t cq = (int64_t)kh * kD + pi, ck = (int64_t)(p.nk + kh) * kD + pi;
    ConvInW<MT> ca, cb;
    GateIn gi{};
    if (tid < kD) {
        conv_load_w(ca, ring, x, p.w, cv, C, p.taps);
        if (tid == 0) gi = gate_load(p, seq, h);
    } else {
        conv_load_w(ca, ring, x, p.w, cq, C, p.taps);
        conv_load_w(cb, ring, x, p.w, ck, C, p.taps);
    }

    // 2. the state loads
    extern __shared__ __align__(16) unsigned char smem_raw[];   // staged: [kD rows][VPR]
    uint4 *mine = reinterpret_cast<uint4 *>(smem_raw) + (row0 + sub) * VPR + (lane % LPR);
    uint4 raw[STAGED ? 1 : (NB > 1 ? 2 : 1)][STAGED ? 1 : PER];
    if constexpr (STAGED) {
#pragma unroll
        for (int gi = 0; gi < kGroups; ++gi) {
#pragma unroll
            for (int ii = 0; ii < PER; ++ii) {
                const int i = gi * PER + ii;
                cp_async16(mine + i * RPL * VPR, rowp + (int64_t)i * RPL * kD);
            }
            cp_async_commit();
        }
    } else {
#pragma unroll
        for (int i = 0; i < PER; ++i) raw[0][i] = ld_stream16(rowp + (int64_t)i * RPL * kD);
    }

    // 3. the producers' arithmetic while the state streams in
    if (tid < kD) {
        v_s[pi] = conv_silu_w(ca, p.taps);
        conv_shift(ca.in, ring + cv, C, p.taps);
        if (tid == 0) gates_of(gi, gate_s[0], gate_s[1]);
    } else {
        const float qv = conv_silu_w(ca, p.taps), kv = conv_silu_w(cb, p.taps);
        conv_shift(ca.in, &ring_new[0][0][pi], kD, p.taps);
        conv_shift(cb.in, &ring_new[1][0][pi], kD, p.taps);
        const float sq = group_sum<32>(qv * qv), sk = group_sum<32>(kv * kv);
        if (lane == 0) { red_q[warp - 4] = sq; red_k[warp - 4] = sk; }
        asm volatile("bar.sync 1, 128;" ::: "memory");  // the four producer warps
        const float tq = (red_q[0] + red_q[1]) + (red_q[2] + red_q[3]);
        const float tk = (red_k[0] + red_k[1]) + (red_k[2] + red_k[3]);
        q_s[pi] = qv / sqrtf(tq + p.l2_eps);
        k_s[pi] = kv / sqrtf(tk + p.l2_eps);
    }
    __syncthreads();                                     // this CTA is done reading the q/k ring rows

    float kx[EPV], qx[EPV];
#pragma unroll
    for (int j = 0; j < EPV; j += 4) {
        const float4 a = *reinterpret_cast<const float4 *>(k_s + col + j);
        const float4 b = *reinterpret_cast<const float4 *>(q_s + col + j);
        kx[j] = a.x; kx[j + 1] = a.y; kx[j + 2] = a.z; kx[j + 3] = a.w;
        qx[j] = b.x; qx[j + 1] = b.y; qx[j + 2] = b.z; qx[j + 3] = b.w;
    }

    const bool row_lane = lane < kRowsPerWarp;
    const float v_l = row_lane ? v_s[row0 + lane] : 0.f;
    float z_l = 0.f, gn_l = 0.f;
    if (row_lane) {
        z_l = __ldg(p.z + seq * p.z_stride + (int64_t)h * kD + row0 + lane);
        gn_l = __ldg(p.gn + row0 + lane);
    }
    const float alpha = gate_s[0], beta = gate_s[1];
    float kq = 0.f;
#pragma unroll
    for (int j = 0; j < EPV; ++j) kq = fmaf(kx[j], qx[j], kq);
    kq = group_sum<LPR>(kq);

    // 4. the step, as in the decode kernel.  fp32: PER rows at once (a commit group or register batch),
    // u and w by one reduce-scatter over the row's lanes (the butterfly's sums bit for bit), then the
    // rows' coefficients broadcast back; fp16 (48 registers a thread hold no group of rows): a row at a
    // time, a butterfly per sum
    constexpr int G = sizeof(TS) == 4 ? PER : 1;
    float o_keep = 0.f;
    auto row_step = [&](const uint4 packed, const int i) {
        float s[EPV];
        V::unpack(packed, s);
        float u = 0.f, w = 0.f;
#pragma unroll
        for (int j = 0; j < EPV; ++j) { u = fmaf(s[j], kx[j], u); w = fmaf(s[j], qx[j], w); }
        u = group_sum<LPR>(u);
        w = group_sum<LPR>(w);
        const float va = __shfl_sync(kFull, v_l, i * RPL + sub);
        const float coef = beta * (va - alpha * u);
        const float oa = (alpha * w + coef * kq) * p.inv_sqrt_d;
#pragma unroll
        for (int j = 0; j < EPV; ++j) s[j] = fmaf(coef, kx[j], alpha * s[j]);
        st_stream16(rowp + (int64_t)i * RPL * kD, V::pack(s));
        if constexpr (RPL == 1) {
            if (lane == i) o_keep = oa;
        } else {
#pragma unroll
            for (int r = 0; r < RPL; ++r) {
                const float orr = __shfl_sync(kFull, oa, r * LPR);
                if (lane == i * RPL + r) o_keep = orr;
            }
        }
    };
    auto group_step = [&](const uint4 (&vec)[G], const int i0) {
        constexpr int R = LPR / (2 * G);
        static_assert(R >= 1 && (G == 1 || G == PER), "a group's 2 G values over the LPR lanes of a row");
        float part[2 * G];
#pragma unroll
        for (int i = 0; i < G; ++i) {
            float s[EPV];
            V::unpack(vec[i], s);
            float u = 0.f, w = 0.f;
#pragma unroll
            for (int j = 0; j < EPV; ++j) { u = fmaf(s[j], kx[j], u); w = fmaf(s[j], qx[j], w); }
            part[2 * i] = u;
            part[2 * i + 1] = w;
        }
        const float mine_sum = reduce_scatter<LPR, 2 * G>(part, lane);
        const float other = __shfl_xor_sync(kFull, mine_sum, R);
        const bool is_w = ((lane % LPR) / R) & 1;
        const float u = is_w ? other : mine_sum, w = is_w ? mine_sum : other;
        const int vi = (lane % LPR) / (2 * R);               // the vector (row) these lanes reduced
        const float va = __shfl_sync(kFull, v_l, (i0 + vi) * RPL + sub);
        const float coef = beta * (va - alpha * u);
        const float oa = (alpha * w + coef * kq) * p.inv_sqrt_d;
        const int gbase = lane & ~(LPR - 1);
        float cf[G];
#pragma unroll
        for (int i = 0; i < G; ++i) cf[i] = __shfl_sync(kFull, coef, gbase + 2 * R * i);
        {   // lane r < kRowsPerWarp keeps the o of row r: vector r / RPL of row group r % RPL
            const int vr = lane / RPL - i0;
            const float ok = __shfl_sync(kFull, oa, (lane % RPL) * LPR + (vr & (G - 1)) * 2 * R);
            if (lane < kRowsPerWarp && vr >= 0 && vr < G) o_keep = ok;
        }
#pragma unroll
        for (int i = 0; i < G; ++i) {
            float s[EPV];
            V::unpack(vec[i], s);
#pragma unroll
            for (int j = 0; j < EPV; ++j) s[j] = fmaf(cf[i], kx[j], alpha * s[j]);
            st_stream16(rowp + (int64_t)(i0 + i) * RPL * kD, V::pack(s));
        }
    };
    // This CTA's reads of the key head's q/k ring rows ended at the __syncthreads after step 3.  It
    // counts itself (fence + atomic add, one thread) as its last batch of rows begins: the fence
    // waits for the counting thread's own memory operations in flight, which by then are that
    // batch's loads (needed next anyway) and the streaming stores of earlier rows, and the add's
    // round trip overlaps the batch.  (Taken
    // right after step 3, the fence held the thread's warp until all its first loads had landed:
    // 38.3 us a launch at batch 32; after the rows, 35.1 us; here, 34.2 us.)  Its result is first
    // needed after the norm's barrier.
    constexpr int kCounter = kWarps * 32 - 1;
    int seen = 0;
    auto count_reader = [&](int bt) {
        if (bt == NBAT - 1 && tid == kCounter) {
            __threadfence();                             // every read of the ring comes before the count
            seen = atomicAdd(p.counters + cl, 1);
        }
    };
#pragma unroll
    for (int bt = 0; bt < NBAT; ++bt) {
        if constexpr (STAGED) {
            if (bt == 0) cp_async_wait<kGroups - 1>();
            else if (bt == 1) cp_async_wait<kGroups - 2>();
            else if (bt == 2) cp_async_wait<kGroups - 3>();
            else cp_async_wait<0>();
            count_reader(bt);
            if constexpr (G > 1) {
                uint4 vec[G];
#pragma unroll
                for (int ii = 0; ii < G; ++ii) vec[ii] = mine[(bt * PER + ii) * RPL * VPR];
                group_step(vec, bt * PER);
            } else {
#pragma unroll
                for (int ii = 0; ii < PER; ++ii) row_step(mine[(bt * PER + ii) * RPL * VPR], bt * PER + ii);
            }
        } else {
            if (bt + 1 < NBAT) {
#pragma unroll
                for (int i = 0; i < PER; ++i)
                    raw[(bt + 1) & 1][i] = ld_stream16(rowp + (int64_t)((bt + 1) * PER + i) * RPL * kD);
            }
            count_reader(bt);
            if constexpr (G > 1) {
                group_step(raw[bt & 1], bt * PER);
            } else {
#pragma unroll
                for (int ii = 0; ii < PER; ++ii) row_step(raw[bt & 1][ii], bt * PER + ii);
            }
        }
    }

    // 5. gated RMS norm over the head's outputs
    const float ss = group_sum<32>(o_keep * o_keep);
    if (lane == 0) red[warp] = ss;
    if (tid == kCounter) {
        const bool last = seen == p.repeat - 1;
        if (last) __threadfence();                       // every other reader's count came first
        last_reader = last;
    }
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) tot += red[i];
    const float rstd = rsqrtf(tot * (1.0f / kD) + p.eps);
    if (row_lane) {
        const float y = gn_l * o_keep * rstd * silu(z_l);
        p.out[seq * p.out_stride + (int64_t)h * kD + row0 + lane] = bf16_bits_rn(y);
    }

    // 6. the last reader of the key head's q/k ring rows writes their new contents
    if (last_reader) {                                   // read after the __syncthreads of step 5
        if (tid >= kD) {
            const int i = tid - kD;
            for (int t = 0; t < p.taps; ++t) {
                ring[(int64_t)t * C + (int64_t)kh * kD + i] = ring_new[0][t][i];
                ring[(int64_t)t * C + (int64_t)(p.nk + kh) * kD + i] = ring_new[1][t][i];
            }
        }
        if (tid == 0) p.counters[cl] = 0;               // ready for the next call
    }
}

// One CTA per (sequence, key head) and its R = NV/NK value heads (the page's
// block shape; taken for fp16 states): q and k are computed once, every ring
// row of the key head is written in place by its only owner (no counter), and
// the value heads are stepped one after another from one 32 KB shared-memory
// buffer: as soon as a lane has stepped a commit group of rows of head r, it
// copies the same rows of head r + 1 into the slots it has just read (a lane
// reads back only its own copies, so no barrier), and the next head streams in
// while this one finishes (150.4 -> 146.3 us at 256 slots; a second 32 KB
// buffer measured slower, with fewer CTAs per SM).  With an fp16 head only 32
// KB, the per-value-head kernel spent more on recomputing the key head's q and
// k three times than on the state stream.
constexpr int kMaxRepeat = 8;

__device__ __forceinline__ void cp_async_wait_n(int n) {
    switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    case 6: cp_async_wait<6>(); break;
    default: cp_async_wait<7>(); break;
    }
}

template <typename TS, int MINB>
__global__ void __launch_bounds__(kWarps * 32, MINB)
conv_norm_kh(const ConvNormParams p)
{
    using V = Vec16<TS>;
    constexpr int EPV = V::N;
    constexpr int LPR = kD / EPV;
    constexpr int RPL = 32 / LPR;
    constexpr int NLD = kRowsPerWarp / RPL;
    constexpr int VPR = kD * (int)sizeof(TS) / 16;
    constexpr int PER = NLD / kGroups;
    static_assert(NLD % kGroups == 0, "shape");

    extern __shared__ __align__(16) unsigned char smem_raw[];   // one head, [kD rows][VPR]
    __shared__ __align__(16) float q_s[kD];
    __shared__ __align__(16) float k_s[kD];
    __shared__ float v_s[kMaxRepeat][kD];
    __shared__ float red_qk[kWarps], red[2][kWarps];
    __shared__ float gate_s[kMaxRepeat][2];

    const int cl = blockIdx.x;                          // (sequence, key head)
    const int seq = cl / p.nk;
    const int kh = cl - seq * p.nk;
    const int R = p.repeat;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sub = lane / LPR;
    const int col = (lane % LPR) * EPV;
    const int row0 = warp * kRowsPerWarp;
    const int64_t C = (int64_t)(2 * p.nk + p.nv) * kD;
    TS *state_seq = reinterpret_cast<TS *>(p.state) + seq * p.pitch;

    auto rowp_of = [&](int r) {
        return state_seq + (int64_t)(kh + r * p.nk) * kD * kD + (int64_t)(row0 + sub) * kD + col;
    };
    uint4 *const mine = reinterpret_cast<uint4 *>(smem_raw) + (row0 + sub) * VPR + (lane % LPR);
    auto issue_group = [&](int r, int gi) {             // commit group gi of head r's rows
        TS *rp = rowp_of(r);
#pragma unroll
        for (int ii = 0; ii < PER; ++ii) {
            const int i = gi * PER + ii;
            cp_async16(mine + i * RPL * VPR, rp + (int64_t)i * RPL * kD);
        }
        cp_async_commit();
    };

    // 1. the first head's state in flight before the producers run
#pragma unroll
    for (int gi = 0; gi < kGroups; ++gi) issue_group(0, gi);

    // 2. producers: q (threads 0..127) and k (128..255) of the key head, then the v channels of its
    //    value heads; this CTA owns every one of these ring rows, so each is shifted in place
    float *ring = p.ring + seq * p.ring_pitch;
    const float *x = p.x + seq * p.x_stride;
    {
        const int i = tid & (kD - 1);
        const int64_t c = tid < kD ? (int64_t)kh * kD + i : (int64_t)(p.nk + kh) * kD + i;
        const float val = conv_silu_channel(ring, x, p.w, c, C, p.taps);
        const float sq = group_sum<32>(val * val);
        if (lane == 0) red_qk[warp] = sq;
        __syncthreads();
        const int w0 = tid < kD ? 0 : 4;
        const float t = (red_qk[w0] + red_qk[w0 + 1]) + (red_qk[w0 + 2] + red_qk[w0 + 3]);
        (tid < kD ? q_s : k_s)[i] = val / sqrtf(t + p.l2_eps);
    }
    for (int j = tid; j < R * kD; j += kWarps * 32) {
        const int r = j / kD, i = j - r * kD;
        v_s[r][i] = conv_silu_channel(ring, x, p.w, 2 * (int64_t)p.nk * kD + (int64_t)(kh + r * p.nk) * kD + i,
                                      C, p.taps);
    }
    if (tid < R) gates(p, seq, kh + tid * p.nk, gate_s[tid][0], gate_s[tid][1]);
    __syncthreads();

    float kx[EPV], qx[EPV];
#pragma unroll
    for (int j = 0; j < EPV; j += 4) {
        const float4 a = *reinterpret_cast<const float4 *>(k_s + col + j);
        const float4 b = *reinterpret_cast<const float4 *>(q_s + col + j);
        kx[j] = a.x; kx[j + 1] = a.y; kx[j + 2] = a.z; kx[j + 3] = a.w;
        qx[j] = b.x; qx[j + 1] = b.y; qx[j + 2] = b.z; qx[j + 3] = b.w;
    }
    float kq = 0.f;
#pragma unroll
    for (int j = 0; j < EPV; ++j) kq = fmaf(kx[j], qx[j], kq);
    kq = group_sum<LPR>(kq);
    const bool row_lane = lane < kRowsPerWarp;
    const float gn_l = row_lane ? __ldg(p.gn + row0 + lane) : 0.f;

    // 3. the value heads in turn
    for (int r = 0; r < R; ++r) {
        const int h = kh + r * p.nk;
        TS *rowp = rowp_of(r);
        const float v_l = row_lane ? v_s[r][row0 + lane] : 0.f;
        const float z_l = row_lane ? __ldg(p.z + seq * p.z_stride + (int64_t)h * kD + row0 + lane) : 0.f;
        const float alpha = gate_s[r][0], beta = gate_s[r][1];
        float o_keep = 0.f;
#pragma unroll
        for (int gi = 0; gi < kGroups; ++gi) {
            if (r + 1 < R) cp_async_wait<kGroups - 1>();   // this group; the next head's earlier ones may pend
            else cp_async_wait_n(kGroups - 1 - gi);
#pragma unroll
            for (int ii = 0; ii < PER; ++ii) {
                const int i = gi * PER + ii;
                float s[EPV];
                V::unpack(mine[i * RPL * VPR], s);
                float u = 0.f, w = 0.f;
#pragma unroll
                for (int j = 0; j < EPV; ++j) { u = fmaf(s[j], kx[j], u); w = fmaf(s[j], qx[j], w); }
                u = group_sum<LPR>(u);
                w = group_sum<LPR>(w);
                const float va = __shfl_sync(kFull, v_l, i * RPL + sub);
                const float coef = beta * (va - alpha * u);
                const float oa = (alpha * w + coef * kq) * p.inv_sqrt_d;
#pragma unroll
                for (int j = 0; j < EPV; ++j) s[j] = fmaf(coef, kx[j], alpha * s[j]);
                st_stream16(rowp + (int64_t)i * RPL * kD, V::pack(s));
                if constexpr (RPL == 1) {
                    if (lane == i) o_keep = oa;
                } else {
#pragma unroll
                    for (int rr = 0; rr < RPL; ++rr) {
                        const float orr = __shfl_sync(kFull, oa, rr * LPR);
                        if (lane == i * RPL + rr) o_keep = orr;
                    }
                }
            }
            if (r + 1 < R) issue_group(r + 1, gi);      // refill the slots just stepped with head r + 1
        }
        const float ss = group_sum<32>(o_keep * o_keep);
        if (lane == 0) red[r & 1][warp] = ss;
        __syncthreads();                                // also: every warp is done with this buffer
        float tot = 0.f;
#pragma unroll
        for (int i = 0; i < kWarps; ++i) tot += red[r & 1][i];
        const float rstd = rsqrtf(tot * (1.0f / kD) + p.eps);
        if (row_lane) {
            const float y = gn_l * o_keep * rstd * silu(z_l);
            p.out[seq * p.out_stride + (int64_t)h * kD + row0 + lane] = bf16_bits_rn(y);
        }
    }
}

// Any 1 <= D <= 256, any alignment, any NV/NK: one CTA per (sequence, key
// head); the producers for the key head and all of its value heads go to
// shared memory, then the value heads are stepped one after the other (warp
// per row) and normed.
constexpr int kGenWarps = 4;
constexpr int kMaxD = 256;

template <typename TS>
__global__ void __launch_bounds__(kGenWarps * 32)
conv_norm_generic(const ConvNormParams p)
{
    constexpr int MAXV = kMaxD / 32;
    extern __shared__ float dyn[];               // q[D], k[D], v[repeat][D], o[D], gates[2 repeat]
    __shared__ float red[kGenWarps], red2[kGenWarps];

    const int D = p.d, R = p.repeat;
    const int seq = blockIdx.x / p.nk;
    const int kh = blockIdx.x - seq * p.nk;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t C = (int64_t)(2 * p.nk + p.nv) * D;
    float *q_s = dyn, *k_s = dyn + D, *v_s = dyn + 2 * D, *o_s = dyn + (2 + R) * D, *g_s = o_s + D;

    float *ring = p.ring + seq * p.ring_pitch;
    const float *x = p.x + seq * p.x_stride;
    for (int i = tid; i < D; i += kGenWarps * 32) {
        q_s[i] = conv_silu_channel(ring, x, p.w, (int64_t)kh * D + i, C, p.taps);
        k_s[i] = conv_silu_channel(ring, x, p.w, (int64_t)(p.nk + kh) * D + i, C, p.taps);
    }
    for (int i = tid; i < R * D; i += kGenWarps * 32) {
        const int r = i / D, j = i - r * D;
        const int h = kh + r * p.nk;
        v_s[i] = conv_silu_channel(ring, x, p.w, 2 * (int64_t)p.nk * D + (int64_t)h * D + j, C, p.taps);
    }
    if (tid < R) gates(p, seq, kh + tid * p.nk, g_s[2 * tid], g_s[2 * tid + 1]);
    __syncthreads();
    {   // L2 of q and k
        float sq = 0.f, sk = 0.f;
        for (int i = tid; i < D; i += kGenWarps * 32) { sq += q_s[i] * q_s[i]; sk += k_s[i] * k_s[i]; }
        sq = group_sum<32>(sq); sk = group_sum<32>(sk);
        if (lane == 0) { red[warp] = sq; red2[warp] = sk; }
        __syncthreads();
        float tq = 0.f, tk = 0.f;
#pragma unroll
        for (int i = 0; i < kGenWarps; ++i) { tq += red[i]; tk += red2[i]; }
        const float dq = sqrtf(tq + p.l2_eps), dk = sqrtf(tk + p.l2_eps);
        __syncthreads();
        for (int i = tid; i < D; i += kGenWarps * 32) { q_s[i] = q_s[i] / dq; k_s[i] = k_s[i] / dk; }
        __syncthreads();
    }
    float kreg[MAXV], qreg[MAXV];
    float kq = 0.f;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
        const int c = lane + 32 * j;
        kreg[j] = c < D ? k_s[c] : 0.f;
        qreg[j] = c < D ? q_s[c] : 0.f;
        kq = fmaf(kreg[j], qreg[j], kq);
    }
    kq = group_sum<32>(kq);

    for (int r = 0; r < R; ++r) {
        const int h = kh + r * p.nk;
        const float alpha = g_s[2 * r], beta = g_s[2 * r + 1];
        TS *S = reinterpret_cast<TS *>(p.state) + seq * p.pitch + (int64_t)h * D * D;
        for (int a = warp; a < D; a += kGenWarps) {
            TS *row = S + (int64_t)a * D;
            float s[MAXV];
            float u = 0.f, w = 0.f;
#pragma unroll
            for (int j = 0; j < MAXV; ++j) {
                const int c = lane + 32 * j;
                s[j] = c < D ? to_f32<TS>(row[c]) : 0.f;
                u = fmaf(s[j], kreg[j], u);
                w = fmaf(s[j], qreg[j], w);
            }
            u = group_sum<32>(u);
            w = group_sum<32>(w);
            const float coef = beta * (v_s[r * D + a] - alpha * u);
            const float oa = (alpha * w + coef * kq) * p.inv_sqrt_d;
#pragma unroll
            for (int j = 0; j < MAXV; ++j) {
                const int c = lane + 32 * j;
                if (c < D) row[c] = from_f32<TS>(fmaf(coef, kreg[j], alpha * s[j]));
            }
            if (lane == 0) o_s[a] = oa;
        }
        __syncthreads();
        float ss = 0.f;
        for (int a = tid; a < D; a += kGenWarps * 32) ss += o_s[a] * o_s[a];
        ss = group_sum<32>(ss);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int i = 0; i < kGenWarps; ++i) tot += red[i];
        const float rstd = rsqrtf(tot / (float)D + p.eps);
        const float *zp = p.z + seq * p.z_stride + (int64_t)h * D;
        uint16_t *op = p.out + seq * p.out_stride + (int64_t)h * D;
        for (int a = tid; a < D; a += kGenWarps * 32)
            op[a] = bf16_bits_rn(p.gn[a] * o_s[a] * rstd * silu(zp[a]));
        __syncthreads();                          // o_s and red reused by the next head
    }
}

// Shapes of the per-value-head D == 128 kernel, by measurement on GB300 (one
// layer at batch 32 fp32, 256-slot fp16 pool): fp32 register batches (4 x 4
// loads, 4 CTAs per SM: a CTA spends part of its life in the producer phase,
// so more of them keep the state streaming; 34.2 us a launch, against 42.4 us
// for 2 x 8 loads at 3 CTAs per SM and 39.3 us staged in shared memory at 3);
// fp16 staged in shared memory (32 KB + 10 KB a CTA, 5 CTAs per SM) -- used
// for fp16 only when NV/NK > 8.
template <typename TS> struct ConvShape {
    static constexpr bool kStaged = false;
    static constexpr int kBatches = 4, kMinBlocks = 4;
};
template <> struct ConvShape<__half> {
    static constexpr bool kStaged = true;
    static constexpr int kBatches = 1, kMinBlocks = 5;
};

// The per-value-head kernel with tap bound MT.
template <typename TS, int MT>
cudaError_t launch_d128(const ConvNormParams &p, cudaStream_t s)
{
    using F = ConvShape<TS>;
    const int dyn = F::kStaged ? stage_bytes<TS>() : 0;
    const unsigned grid = (unsigned)((int64_t)p.batch * p.nv);
    // early launch (grids of a few waves) with the whole head asked of the L2: these CTAs run
    // the conv and gate producers before they need the state (measured: whole 32.6 us, half 34.3)
    if (early_grid(grid, F::kMinBlocks)) {
        ConvNormParams q = p;
        q.pf_bytes = (unsigned)(kD * kD * sizeof(TS));
        constexpr auto kern = conv_norm_d128<TS, F::kStaged, F::kBatches, F::kMinBlocks, true, MT>;
        if (F::kStaged) {
            const cudaError_t e = allow_dynamic_smem<kern>(dyn);
            if (e != cudaSuccess) return e;
        }
        return launch_early(kern, grid, kWarps * 32, dyn, s, true, q);
    }
    constexpr auto kern = conv_norm_d128<TS, F::kStaged, F::kBatches, F::kMinBlocks, false, MT>;
    if (F::kStaged) {
        const cudaError_t e = allow_dynamic_smem<kern>(dyn);
        if (e != cudaSuccess) return e;
    }
    return launch_early(kern, grid, kWarps * 32, dyn, s, false, p);
}

template <typename TS>
cudaError_t launch_typed(const ConvNormParams &p, bool fast, cudaStream_t s)
{
    if constexpr (sizeof(TS) == 2) {
        if (fast && p.repeat <= kMaxRepeat) {            // one CTA per key head, one staging buffer
            constexpr auto kern = conv_norm_kh<TS, 5>;
            const cudaError_t e = allow_dynamic_smem<kern>(stage_bytes<TS>());
            if (e != cudaSuccess) return e;
            // a plain launch: launched early (with or without an L2 prefetch of its heads) it
            // measured no faster at 256 slots
            kern<<<(unsigned)((int64_t)p.batch * p.nk), kWarps * 32, stage_bytes<TS>(), s>>>(p);
            return cudaGetLastError();
        }
    }
    if (fast) return p.taps <= 4 ? launch_d128<TS, 4>(p, s) : launch_d128<TS, kMaxTaps>(p, s);
    const size_t smem = sizeof(float) * ((size_t)(3 + p.repeat) * p.d + 2 * (size_t)p.repeat);
    conv_norm_generic<TS><<<(unsigned)((int64_t)p.batch * p.nk), kGenWarps * 32, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_conv_norm(const ConvNormParams &p, bool f16_state, bool fast, cudaStream_t s)
{
    return f16_state ? launch_typed<__half>(p, fast, s) : launch_typed<float>(p, fast, s);
}

}  // namespace gdn
