// gdn_chunk2.cu -- two tokens through the gated delta rule in one launch (the
// verify step of speculative decoding), writing the state after the first
// token to a second buffer so a rejected draft token can be rolled back.
//
// Follows metrale_model_layers/layers/ops/ssm_gdn_a.rs, launcher
// `gdn_decode_chunk2` (two tokens per launch, the intermediate state written
// for rollback, strides in elements); the step is
// logicaffeine_compile/codegen_cuda/gdn.rs, kernel `gdn_step`.
//
// Per row the arithmetic is exactly that of the single-token kernels in
// gdn_decode.cu, applied twice with the row slice kept in registers: the state
// is read once and written twice (intermediate + final), instead of read twice
// and written twice by two launches.  With an fp16 state the row is rounded to
// fp16 after the first token and the second token continues from the rounded
// values, so the result is bitwise the one two single-token calls give.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kD = 128;

// STAGED: the head goes to shared memory by cp.async with every load in flight
// (kGroups commit groups, each consumed as it lands); otherwise NB register
// batches, the next in flight while one is stepped.  Shapes by measurement on
// GB300 (batch 32 fp32 over 8 layers' states, the 256-slot fp16 pool; all
// bitwise-identical): fp16 staged at 4 CTAs/SM 192.9 us against register
// batches (8 warps x 2 x 3 CTAs/SM) 207.5 and staged at 3 CTAs/SM 209.9; fp32
// staged at 3 CTAs/SM 47.7 us against register batches (8 x 4 x 4) 47.9.
constexpr int kGroups = 4;
template <typename TS> struct Chunk2Shape {
    static constexpr bool kStaged = true;
    static constexpr int kWarps = 8, kBatches = 1, kMinBlocks = 3;
};
template <> struct Chunk2Shape<__half> {
    static constexpr bool kStaged = true;
    static constexpr int kWarps = 8, kBatches = 1, kMinBlocks = 4;
};

template <typename TS>
constexpr int stage_bytes() { return kD * kD * (int)sizeof(TS); }

template <typename TS, int WARPS, bool STAGED, int NB, int MINB, bool EARLY>
__global__ void __launch_bounds__(WARPS * 32, MINB)
chunk2_d128(const DecodeParams p)
{
    using V = Vec16<TS>;
    constexpr int EPV = V::N;                  // state elements per 16-byte vector
    constexpr int LPR = kD / EPV;              // lanes per state row: 32 fp32, 16 fp16
    constexpr int RPL = 32 / LPR;              // rows per warp-wide load
    constexpr int RPW = kD / WARPS;            // rows per warp
    constexpr int NLD = RPW / RPL;             // 16-byte state loads per lane
    constexpr int VPR = kD * (int)sizeof(TS) / 16;   // 16-byte vectors per state row
    constexpr int NBAT = STAGED ? kGroups : NB;      // groups / batches of loads
    constexpr int LPB = NLD / NBAT;                  // loads per group / batch
    static_assert(RPW <= 32 && NLD % NBAT == 0, "shape");

    const int unit = blockIdx.x;               // (sequence, value head)
    const int seq = unit / p.nv;
    const int h = unit - seq * p.nv;
    const int g = h % p.nk;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR;
    const int col = (lane % LPR) * EPV;
    const int row0 = warp * RPW;
    const int64_t slice = (int64_t)h * kD * kD + (int64_t)(row0 + sub) * kD + col;

    TS *rowp = reinterpret_cast<TS *>(p.state) + seq * p.pitch + slice;
    TS *midp = reinterpret_cast<TS *>(p.state_mid) + seq * p.mid_pitch + slice;
    early_start<EARLY>(reinterpret_cast<TS *>(p.state) + seq * p.pitch + (int64_t)h * kD * kD, p.pf_bytes);

    extern __shared__ __align__(16) unsigned char smem_raw[];   // staged: [kD rows][VPR], the head as stored
    uint4 *mine = reinterpret_cast<uint4 *>(smem_raw) + (row0 + sub) * VPR + (lane % LPR);
    uint4 raw[STAGED ? 1 : (NB > 1 ? 2 : 1)][STAGED ? 1 : LPB];
    if constexpr (STAGED) {                    // a lane reads back only what it copied: no barrier
#pragma unroll
        for (int gi = 0; gi < kGroups; ++gi) {
#pragma unroll
            for (int ii = 0; ii < LPB; ++ii) {
                const int i = gi * LPB + ii;
                cp_async16(mine + i * RPL * VPR, rowp + (int64_t)i * RPL * kD);
            }
            cp_async_commit();
        }
    } else {
#pragma unroll
        for (int i = 0; i < LPB; ++i) raw[0][i] = ld_stream16(rowp + (int64_t)i * RPL * kD);
    }

    // token t of sequence b reads input row 2 b + t
    const bool row_lane = lane < RPW;
    float kx[2][EPV], qx[2][EPV], v_l[2], alpha[2], beta[2], kq[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int64_t row = (int64_t)seq * 2 + t;
        const float *kp = p.k + row * p.qk_stride + (int64_t)g * kD + col;
        const float *qp = p.q + row * p.qk_stride + (int64_t)g * kD + col;
#pragma unroll
        for (int j = 0; j < EPV; j += 4) {
            const float4 a = ld_ro_f4(kp + j), b = ld_ro_f4(qp + j);
            kx[t][j] = a.x; kx[t][j + 1] = a.y; kx[t][j + 2] = a.z; kx[t][j + 3] = a.w;
            qx[t][j] = b.x; qx[t][j + 1] = b.y; qx[t][j + 2] = b.z; qx[t][j + 3] = b.w;
        }
        v_l[t] = row_lane ? __ldg(p.v + row * p.v_stride + (int64_t)h * kD + row0 + lane) : 0.f;
        alpha[t] = __ldg(p.alpha + row * p.gb_stride + h);
        beta[t] = __ldg(p.beta + row * p.gb_stride + h);
        float a = 0.f;
#pragma unroll
        for (int j = 0; j < EPV; ++j) a = fmaf(kx[t][j], qx[t][j], a);
        kq[t] = group_sum<LPR>(a);
    }

    float o_keep[2] = {0.f, 0.f};
    // fp32: LPB rows at once (a commit group or a register batch), token after token: u and w of the
    // rows by one reduce-scatter over the row's lanes (the butterfly's sums bit for bit, as in the
    // single-token kernel), the rows' coefficients broadcast back; token 1 continues from the state
    // as stored after token 0.  fp16 (64 registers a thread, with both tokens' k and q, hold no group
    // of rows): a row at a time, a butterfly per sum -- a one-row group measured 1.4 % slower (its
    // shuffles form one longer chain instead of two interleaved ones).
    constexpr int G = sizeof(TS) == 4 ? LPB : 1;
    auto row_steps = [&](const uint4 packed_in, const int i) {   // both tokens on state row slice i
            float s[EPV];
            V::unpack(packed_in, s);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                float u = 0.f, w = 0.f;
#pragma unroll
                for (int j = 0; j < EPV; ++j) { u = fmaf(s[j], kx[t][j], u); w = fmaf(s[j], qx[t][j], w); }
                u = group_sum<LPR>(u);
                w = group_sum<LPR>(w);
                const float va = __shfl_sync(kFull, v_l[t], i * RPL + sub);
                const float coef = beta[t] * (va - alpha[t] * u);
                const float oa = (alpha[t] * w + coef * kq[t]) * p.inv_sqrt_d;
#pragma unroll
                for (int j = 0; j < EPV; ++j) s[j] = fmaf(coef, kx[t][j], alpha[t] * s[j]);
                const uint4 packed = V::pack(s);
                if (t == 0) {
                    st_stream16(midp + (int64_t)i * RPL * kD, packed);
                    V::unpack(packed, s);      // continue from the stored (rounded) state
                } else {
                    st_stream16(rowp + (int64_t)i * RPL * kD, packed);
                }
                if constexpr (RPL == 1) {
                    if (lane == i) o_keep[t] = oa;
                } else {
#pragma unroll
                    for (int r = 0; r < RPL; ++r) {
                        const float orr = __shfl_sync(kFull, oa, r * LPR);
                        if (lane == i * RPL + r) o_keep[t] = orr;
                    }
                }
            }
    };
    auto group_steps = [&](const uint4 (&vec)[G], const int i0) {
        constexpr int R = LPR / (2 * G);
        static_assert(R >= 1 && (G == 1 || G == LPB), "a group's 2 G values over the LPR lanes of a row");
        float s[G][EPV];                                     // the rows, unpacked once
#pragma unroll
        for (int ii = 0; ii < G; ++ii) V::unpack(vec[ii], s[ii]);
        const int vi = (lane % LPR) / (2 * R);               // the vector (row) these lanes reduce
        const bool is_w = ((lane % LPR) / R) & 1;
        const int gbase = lane & ~(LPR - 1);
        const int vr = lane / RPL - i0;                      // lane r < RPW keeps row r's o
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            float part[2 * G];
#pragma unroll
            for (int ii = 0; ii < G; ++ii) {
                float u = 0.f, w = 0.f;
#pragma unroll
                for (int j = 0; j < EPV; ++j) { u = fmaf(s[ii][j], kx[t][j], u); w = fmaf(s[ii][j], qx[t][j], w); }
                part[2 * ii] = u;
                part[2 * ii + 1] = w;
            }
            const float mine_sum = reduce_scatter<LPR, 2 * G>(part, lane);
            const float other = __shfl_xor_sync(kFull, mine_sum, R);
            const float u = is_w ? other : mine_sum, w = is_w ? mine_sum : other;
            const float va = __shfl_sync(kFull, v_l[t], (i0 + vi) * RPL + sub);
            const float coef = beta[t] * (va - alpha[t] * u);
            const float oa = (alpha[t] * w + coef * kq[t]) * p.inv_sqrt_d;
            float cf[G];
#pragma unroll
            for (int ii = 0; ii < G; ++ii) cf[ii] = __shfl_sync(kFull, coef, gbase + 2 * R * ii);
            const float ok = __shfl_sync(kFull, oa, (lane % RPL) * LPR + (vr & (G - 1)) * 2 * R);
            if (lane < RPW && vr >= 0 && vr < G) o_keep[t] = ok;
#pragma unroll
            for (int ii = 0; ii < G; ++ii) {
#pragma unroll
                for (int j = 0; j < EPV; ++j) s[ii][j] = fmaf(cf[ii], kx[t][j], alpha[t] * s[ii][j]);
                const uint4 packed = V::pack(s[ii]);
                if (t == 0) {
                    st_stream16(midp + (int64_t)(i0 + ii) * RPL * kD, packed);
                    V::unpack(packed, s[ii]);        // continue from the stored (rounded) state
                } else {
                    st_stream16(rowp + (int64_t)(i0 + ii) * RPL * kD, packed);
                }
            }
        }
    };
#pragma unroll
    for (int bt = 0; bt < NBAT; ++bt) {
        if constexpr (STAGED) {
            if (bt == 0) cp_async_wait<kGroups - 1>();
            else if (bt == 1) cp_async_wait<kGroups - 2>();
            else if (bt == 2) cp_async_wait<kGroups - 3>();
            else cp_async_wait<0>();
            if constexpr (G > 1) {
                uint4 vec[G];
#pragma unroll
                for (int ii = 0; ii < G; ++ii) vec[ii] = mine[(bt * LPB + ii) * RPL * VPR];
                group_steps(vec, bt * LPB);
            } else {
#pragma unroll
                for (int ii = 0; ii < LPB; ++ii) row_steps(mine[(bt * LPB + ii) * RPL * VPR], bt * LPB + ii);
            }
        } else {
            if (bt + 1 < NBAT) {
#pragma unroll
                for (int i = 0; i < LPB; ++i)
                    raw[(bt + 1) & 1][i] = ld_stream16(rowp + (int64_t)((bt + 1) * LPB + i) * RPL * kD);
            }
            if constexpr (G > 1) {
                group_steps(raw[bt & 1], bt * LPB);
            } else {
#pragma unroll
                for (int ii = 0; ii < LPB; ++ii) row_steps(raw[bt & 1][ii], bt * LPB + ii);
            }
        }
    }
    if (row_lane) {
#pragma unroll
        for (int t = 0; t < 2; ++t)
            p.o[((int64_t)seq * 2 + t) * p.o_stride + (int64_t)h * kD + row0 + lane] = o_keep[t];
    }
}

// Any D <= 256 and any alignment: the general single-token kernel's per-row
// arithmetic, applied twice.
constexpr int kGenWarps = 4;
constexpr int kMaxD = 256;

template <typename TS>
__global__ void __launch_bounds__(kGenWarps * 32)
chunk2_generic(const DecodeParams p)
{
    constexpr int MAXV = kMaxD / 32;
    __shared__ float o_s[2][kMaxD];

    const int D = p.d;
    const int seq = blockIdx.x / p.nv;
    const int h = blockIdx.x - seq * p.nv;
    const int g = h % p.nk;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    TS *S = reinterpret_cast<TS *>(p.state) + seq * p.pitch + (int64_t)h * D * D;
    TS *M = reinterpret_cast<TS *>(p.state_mid) + seq * p.mid_pitch + (int64_t)h * D * D;
    const float *vp[2];
    float alpha[2], beta[2], kq[2], kreg[2][MAXV], qreg[2][MAXV];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int64_t row = (int64_t)seq * 2 + t;
        const float *kp = p.k + row * p.qk_stride + (int64_t)g * D;
        const float *qp = p.q + row * p.qk_stride + (int64_t)g * D;
        vp[t] = p.v + row * p.v_stride + (int64_t)h * D;
        alpha[t] = p.alpha[row * p.gb_stride + h];
        beta[t] = p.beta[row * p.gb_stride + h];
        float a = 0.f;
#pragma unroll
        for (int j = 0; j < MAXV; ++j) {
            const int c = lane + 32 * j;
            kreg[t][j] = c < D ? kp[c] : 0.f;
            qreg[t][j] = c < D ? qp[c] : 0.f;
            a = fmaf(kreg[t][j], qreg[t][j], a);
        }
        kq[t] = group_sum<32>(a);
    }

    for (int a = warp; a < D; a += kGenWarps) {
        float s[MAXV];
#pragma unroll
        for (int j = 0; j < MAXV; ++j) {
            const int c = lane + 32 * j;
            s[j] = c < D ? to_f32<TS>(S[(int64_t)a * D + c]) : 0.f;
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            float u = 0.f, w = 0.f;
#pragma unroll
            for (int j = 0; j < MAXV; ++j) {
                u = fmaf(s[j], kreg[t][j], u);
                w = fmaf(s[j], qreg[t][j], w);
            }
            u = group_sum<32>(u);
            w = group_sum<32>(w);
            const float coef = beta[t] * (vp[t][a] - alpha[t] * u);
            const float oa = (alpha[t] * w + coef * kq[t]) * p.inv_sqrt_d;
            TS *dst = (t == 0 ? M : S) + (int64_t)a * D;
#pragma unroll
            for (int j = 0; j < MAXV; ++j) {
                const int c = lane + 32 * j;
                const TS st = from_f32<TS>(fmaf(coef, kreg[t][j], alpha[t] * s[j]));
                s[j] = c < D ? to_f32<TS>(st) : 0.f;   // continue from the stored value
                if (c < D) dst[c] = st;
            }
            if (lane == 0) o_s[t][a] = oa;
        }
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < 2; ++t)
        for (int a = threadIdx.x; a < D; a += kGenWarps * 32)
            p.o[((int64_t)seq * 2 + t) * p.o_stride + (int64_t)h * D + a] = o_s[t][a];
}

template <typename TS>
cudaError_t launch_typed(const DecodeParams &p, bool fast, cudaStream_t s)
{
    const unsigned grid = (unsigned)((int64_t)p.batch * p.nv);
    using F = Chunk2Shape<TS>;
    if (fast) {   // early launch (grids of a few waves) with a quarter of the head asked of the L2
        const int smem = F::kStaged ? stage_bytes<TS>() : 0;
        if (early_grid(grid, F::kMinBlocks)) {
            constexpr auto kern = chunk2_d128<TS, F::kWarps, F::kStaged, F::kBatches, F::kMinBlocks, true>;
            if (F::kStaged) {
                const cudaError_t e = allow_dynamic_smem<kern>(smem);
                if (e != cudaSuccess) return e;
            }
            DecodeParams q = p;
            q.pf_bytes = (unsigned)(kD * kD * sizeof(TS) / 4);
            return launch_early(kern, grid, F::kWarps * 32, smem, s, true, q);
        }
        constexpr auto kern = chunk2_d128<TS, F::kWarps, F::kStaged, F::kBatches, F::kMinBlocks, false>;
        if (F::kStaged) {
            const cudaError_t e = allow_dynamic_smem<kern>(smem);
            if (e != cudaSuccess) return e;
        }
        return launch_early(kern, grid, F::kWarps * 32, smem, s, false, p);
    }
    chunk2_generic<TS><<<grid, kGenWarps * 32, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_chunk2(const DecodeParams &p, bool f16_state, bool fast, cudaStream_t s)
{
    return f16_state ? launch_typed<__half>(p, fast, s) : launch_typed<float>(p, fast, s);
}

}  // namespace gdn
