// kda_recurrent.cu -- token-serial KDA mixer step: single-token decode and multi-token draft
// verify (and the same loop over a whole prompt).
//
// One CTA of 256 threads owns one (sequence, head) tile: the 128 x 128 recurrent state S of
// that head, held in registers in FP32 for the whole launch whatever the storage dtype.
// Per token it fuses, in this order ("KDA fuses the f_b projection, convolution, FP32 recurrence
// and gated output normalization", NVFP4 Kimi K3 targets page, Description):
//   f_b projection (W_fb[h] . f_a, 16 lanes per W row, shuffle-reduced) -> decay alpha;
//   short causal conv + SiLU on the q, k, v channels of the head (window in registers);
//   q, k L2 norms, k.q and beta (warp reductions);
//   decay, S^T k and S^T q in one sweep over the register tile (cross-warp reduce in smem);
//   u = v - S^T k, o = S^T q + beta u (k.q) = (updated S)^T q, gated RMSNorm of o;
//   rank-1 update S += beta k u^T.
// State traffic is one coalesced 128-bit load and store per 16 bytes of the tile: a warp covers
// one 512-byte FP32 row (or two 256-byte BF16 rows) per instruction.  The tile loads are issued
// before the gate math of the first token so that they are in flight while it runs.
//
// Verify ("FP32 per-token draft records with either SSM storage dtype", same page; per-token
// KDA verify states, Kimi K3 on modeling_v2 page, section 5) writes the FP32 state and the conv
// window after every token and leaves the slot untouched; decode / token-serial prefill write
// the final state (rounded once to the storage dtype) and window back to the slot.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int NT = 256;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float softplusf_(float x) { return x > 20.0f ? x : log1pf(expf(x)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

template <int W>
__device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Register tile: a thread owns columns [col, col+VEC) of rows row0 + RPP*p, p < NP.
template <typename ST>
struct Tile {
    static constexpr int VEC = 16 / sizeof(ST);   // 4 (fp32) or 8 (bf16) columns per thread
    static constexpr int TPR = kDv / VEC;          // threads per row: 32 or 16
    static constexpr int RPP = NT / TPR;           // rows per pass: 8 or 16
    static constexpr int NP = kDk / RPP;           // passes: 16 or 8
};

template <typename ST>
__device__ __forceinline__ void unpack(const uint4 &r, float *f);

template <>
__device__ __forceinline__ void unpack<float>(const uint4 &r, float *f)
{
    f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
}

template <>
__device__ __forceinline__ void unpack<__nv_bfloat16>(const uint4 &r, float *f)
{
    f[0] = bf16_lo(r.x); f[1] = bf16_hi(r.x); f[2] = bf16_lo(r.y); f[3] = bf16_hi(r.y);
    f[4] = bf16_lo(r.z); f[5] = bf16_hi(r.z); f[6] = bf16_lo(r.w); f[7] = bf16_hi(r.w);
}

template <typename ST>
__device__ __forceinline__ uint4 pack(const float *f);

template <>
__device__ __forceinline__ uint4 pack<float>(const float *f)
{
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
}

template <>
__device__ __forceinline__ uint4 pack<__nv_bfloat16>(const float *f)
{
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

struct __align__(16) Smem {
    float alpha[kDk];
    float q[kDk];
    float k[kDk];
    float v[kDv];
    float u[kDv];
    float red[NT / 32][2][kDv];   // per-warp partial S^T k / S^T q
    float part[8];                // |q|^2, |k|^2, q.k, -, RMS partials of warps 0..3
    float beta;
};

// Per-thread state of the short convolution: item 0 is q channel tid (tid < 128) or k channel
// tid - 128; item 1 is v channel tid (tid < 128 only).  The window holds the last three
// pre-conv inputs of the channel, oldest first, exactly as stored in the pool.
struct ConvItems {
    int n;
    int tensor[2];
    int ch[2];
    float w[2][kConv];
    __nv_bfloat16 win[2][kTaps];
};

// Gate phase of one token: f_b projection and decay, conv + SiLU, norms, beta -> shared memory.
// Ends with a __syncthreads(); on return sm.alpha/q/k/v/part/beta are valid.
template <bool RECORDS>
__device__ __forceinline__ void gate_phase(const RecurrentParams &p, Smem &sm, ConvItems &cv,
                                           size_t tok, int h, float a_h)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, H = p.H, HC = H * kDk;
    // a1, a2: half-warp hw owns W rows hw + 16 m (m < 8); lane li owns r in [8 li, 8 li + 8)
    {
        const int hw = tid >> 4, li = tid & 15;
        const uint4 fr = *reinterpret_cast<const uint4 *>(p.f_a + tok * kRank + li * 8);
        float fa[8];
        fa[0] = bf16_lo(fr.x); fa[1] = bf16_hi(fr.x); fa[2] = bf16_lo(fr.y); fa[3] = bf16_hi(fr.y);
        fa[4] = bf16_lo(fr.z); fa[5] = bf16_hi(fr.z); fa[6] = bf16_lo(fr.w); fa[7] = bf16_hi(fr.w);
        float mine = 0.f;
#pragma unroll
        for (int m = 0; m < 8; m++) {
            const int i = hw + 16 * m;
            const uint4 wr = __ldg(reinterpret_cast<const uint4 *>(p.W_fb + ((size_t)h * kDk + i) * kRank + li * 8));
            float acc = bf16_lo(wr.x) * fa[0];
            acc = fmaf(bf16_hi(wr.x), fa[1], acc);
            acc = fmaf(bf16_lo(wr.y), fa[2], acc);
            acc = fmaf(bf16_hi(wr.y), fa[3], acc);
            acc = fmaf(bf16_lo(wr.z), fa[4], acc);
            acc = fmaf(bf16_hi(wr.z), fa[5], acc);
            acc = fmaf(bf16_lo(wr.w), fa[6], acc);
            acc = fmaf(bf16_hi(wr.w), fa[7], acc);
            acc = group_sum<16>(acc);
            if (li == m) mine = acc;
        }
        if (li < 8) {
            const int i = hw + 16 * li;
            sm.alpha[i] = expf(-a_h * softplusf_(mine + p.dt_bias[h * kDk + i]));
        }
    }
    // a4: short causal conv + SiLU, window shift; verify records the window after the token
#pragma unroll
    for (int it = 0; it < 2; it++) {
        if (it < cv.n) {
            const int tens = cv.tensor[it], ch = cv.ch[it];
            const __nv_bfloat16 *src = tens == 0 ? p.q : (tens == 1 ? p.k : p.v);
            const __nv_bfloat16 x = src[tok * HC + ch];
            float acc = cv.w[it][0] * bf2f(cv.win[it][0]);
            acc = fmaf(cv.w[it][1], bf2f(cv.win[it][1]), acc);
            acc = fmaf(cv.w[it][2], bf2f(cv.win[it][2]), acc);
            acc = fmaf(cv.w[it][3], bf2f(x), acc);
            const float y = acc / (1.0f + expf(-acc));
            cv.win[it][0] = cv.win[it][1];
            cv.win[it][1] = cv.win[it][2];
            cv.win[it][2] = x;
            const int c = ch - h * kDk;
            if (tens == 0) sm.q[c] = y; else if (tens == 1) sm.k[c] = y; else sm.v[c] = y;
            if (RECORDS) {
#pragma unroll
                for (int j = 0; j < kTaps; j++)
                    p.rec_conv[((tok * 3 + tens) * kTaps + j) * HC + ch] = cv.win[it][j];
            }
        }
    }
    __syncthreads();
    // a3, a5: |q|^2, |k|^2, q.k (raw) and beta
    if (warp < 3) {
        const float4 a = *reinterpret_cast<const float4 *>((warp == 1 ? sm.k : sm.q) + lane * 4);
        const float4 c = *reinterpret_cast<const float4 *>((warp == 0 ? sm.q : sm.k) + lane * 4);
        float s = a.x * c.x + a.y * c.y + a.z * c.z + a.w * c.w;
        s = group_sum<32>(s);
        if (lane == 0) sm.part[warp] = s;
    } else if (tid == 96) {
        sm.beta = sigmoidf_(bf2f(p.beta[tok * H + h]));
    }
    __syncthreads();
}

template <typename ST, bool RECORDS>
__global__ void __launch_bounds__(NT, 2) kda_recurrent_kernel(const RecurrentParams p)
{
    using TL = Tile<ST>;
    constexpr int VEC = TL::VEC, TPR = TL::TPR, RPP = TL::RPP, NP = TL::NP;
    __shared__ Smem sm;

    const int h = blockIdx.x, b = blockIdx.y, H = p.H, HC = H * kDk;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int slot = p.slot_ids[b];
    if (slot < 0 || slot >= p.num_slots) {
        if (tid == 0) atomicOr(p.err_word, KDA_DEVERR_SLOT);
        return;
    }

    const int col = (tid % TPR) * VEC, row0 = tid / TPR;
    ST *tile = reinterpret_cast<ST *>(p.state) + ((size_t)slot * H + h) * (kDk * kDv);
    float s[NP][VEC];

    ConvItems cv;
    cv.n = tid < kDv ? 2 : 1;
    cv.tensor[0] = tid < kDk ? 0 : 1;
    cv.ch[0] = h * kDk + (tid & (kDk - 1));
    cv.tensor[1] = 2;
    cv.ch[1] = h * kDv + (tid & (kDv - 1));

    const float a_h = expf(p.A_log[h]);
    const float q_scale = rsqrtf((float)kDk);

    {
        // issue the tile loads first; they land while the first token's gates are computed
        uint4 raw[NP];
#pragma unroll
        for (int pp = 0; pp < NP; pp++)
            raw[pp] = __ldcs(reinterpret_cast<const uint4 *>(tile + (size_t)(row0 + RPP * pp) * kDv + col));
#pragma unroll
        for (int it = 0; it < 2; it++) {
            if (it < cv.n) {
                const int tens = cv.tensor[it], ch = cv.ch[it];
                const uint2 w = *reinterpret_cast<const uint2 *>(p.conv_w + ((size_t)tens * HC + ch) * kConv);
                cv.w[it][0] = bf16_lo(w.x); cv.w[it][1] = bf16_hi(w.x);
                cv.w[it][2] = bf16_lo(w.y); cv.w[it][3] = bf16_hi(w.y);
#pragma unroll
                for (int j = 0; j < kTaps; j++)
                    cv.win[it][j] = p.conv_state[(((size_t)slot * 3 + tens) * kTaps + j) * HC + ch];
            }
        }
        gate_phase<RECORDS>(p, sm, cv, (size_t)b * p.T, h, a_h);
#pragma unroll
        for (int pp = 0; pp < NP; pp++) unpack<ST>(raw[pp], s[pp]);
    }

    for (int t = 0; t < p.T; t++) {
        const size_t tok = (size_t)b * p.T + t;
        if (t > 0) {
            __syncthreads();   // every reader of the previous token's sm.* is done
            gate_phase<RECORDS>(p, sm, cv, tok, h, a_h);
        }
        const float rq = q_scale / sqrtf(sm.part[0] + p.l2_eps);
        const float rk = 1.0f / sqrtf(sm.part[1] + p.l2_eps);
        const float kq = sm.part[2] * rq * rk;
        const float beta = sm.beta;

        // ---- a6: decay, then S^T k and S^T q in one sweep over the tile
        float ak[VEC], aq[VEC];
#pragma unroll
        for (int c = 0; c < VEC; c++) ak[c] = aq[c] = 0.f;
#pragma unroll
        for (int pp = 0; pp < NP; pp++) {
            const int i = row0 + RPP * pp;
            const float a = sm.alpha[i], kk = sm.k[i] * rk, qq = sm.q[i] * rq;
#pragma unroll
            for (int c = 0; c < VEC; c++) {
                s[pp][c] *= a;
                ak[c] = fmaf(s[pp][c], kk, ak[c]);
                aq[c] = fmaf(s[pp][c], qq, aq[c]);
            }
        }
        if (TPR == 16) {
#pragma unroll
            for (int c = 0; c < VEC; c++) {
                ak[c] += __shfl_xor_sync(0xffffffffu, ak[c], 16);
                aq[c] += __shfl_xor_sync(0xffffffffu, aq[c], 16);
            }
        }
        if (lane < TPR) {
#pragma unroll
            for (int c = 0; c < VEC; c += 4) {
                *reinterpret_cast<float4 *>(&sm.red[warp][0][col + c]) = make_float4(ak[c], ak[c + 1], ak[c + 2], ak[c + 3]);
                *reinterpret_cast<float4 *>(&sm.red[warp][1][col + c]) = make_float4(aq[c], aq[c + 1], aq[c + 2], aq[c + 3]);
            }
        }
        __syncthreads();

        // ---- u = v - S^T k;  o = S^T q + beta u (k.q);  RMS partial sums (a6, a7)
        float o = 0.f;
        if (tid < kDv) {
            float stk = 0.f, stq = 0.f;
#pragma unroll
            for (int w = 0; w < NT / 32; w++) { stk += sm.red[w][0][tid]; stq += sm.red[w][1][tid]; }
            const float u = sm.v[tid] - stk;
            o = stq + beta * u * kq;
            sm.u[tid] = u;
            const float ss = group_sum<32>(o * o);
            if (lane == 0) sm.part[4 + warp] = ss;
        }
        __syncthreads();
        if (tid < kDv) {
            const float ms = (sm.part[4] + sm.part[5] + sm.part[6] + sm.part[7]) * (1.0f / kDv);
            const size_t oi = tok * (size_t)(H * kDv) + (size_t)h * kDv + tid;
            const float y = o * rsqrtf(ms + p.norm_eps) * p.norm_w[tid] * sigmoidf_(bf2f(p.gate[oi]));
            p.out[oi] = __float2bfloat16_rn(y);
        }

        // ---- rank-1 update S += beta k u^T (registers); verify records the FP32 state
        float uu[VEC];
#pragma unroll
        for (int c = 0; c < VEC; c += 4) {
            const float4 u4 = *reinterpret_cast<const float4 *>(&sm.u[col + c]);
            uu[c] = u4.x; uu[c + 1] = u4.y; uu[c + 2] = u4.z; uu[c + 3] = u4.w;
        }
        float *rec = RECORDS ? p.rec_state + (tok * H + h) * (size_t)(kDk * kDv) : nullptr;
#pragma unroll
        for (int pp = 0; pp < NP; pp++) {
            const int i = row0 + RPP * pp;
            const float bk = beta * sm.k[i] * rk;
#pragma unroll
            for (int c = 0; c < VEC; c++) s[pp][c] = fmaf(bk, uu[c], s[pp][c]);
            if (RECORDS) {
#pragma unroll
                for (int c = 0; c < VEC; c += 4)
                    __stcs(reinterpret_cast<float4 *>(rec + (size_t)i * kDv + col + c),
                           make_float4(s[pp][c], s[pp][c + 1], s[pp][c + 2], s[pp][c + 3]));
            }
        }
    }

    if (!RECORDS) {
        // write the state (one rounding to the storage dtype) and the conv window back
#pragma unroll
        for (int pp = 0; pp < NP; pp++)
            __stcs(reinterpret_cast<uint4 *>(tile + (size_t)(row0 + RPP * pp) * kDv + col), pack<ST>(s[pp]));
#pragma unroll
        for (int it = 0; it < 2; it++) {
            if (it < cv.n) {
#pragma unroll
                for (int j = 0; j < kTaps; j++)
                    p.conv_state[(((size_t)slot * 3 + cv.tensor[it]) * kTaps + j) * HC + cv.ch[it]] = cv.win[it][j];
            }
        }
    }
}

}  // namespace

cudaError_t launch_recurrent(const RecurrentParams &p, bool bf16_state, bool records,
                             cudaStream_t stream)
{
    const dim3 grid((unsigned)p.H, (unsigned)p.B), block(NT);
    if (bf16_state) {
        if (records) kda_recurrent_kernel<__nv_bfloat16, true><<<grid, block, 0, stream>>>(p);
        else kda_recurrent_kernel<__nv_bfloat16, false><<<grid, block, 0, stream>>>(p);
    } else {
        if (records) kda_recurrent_kernel<float, true><<<grid, block, 0, stream>>>(p);
        else kda_recurrent_kernel<float, false><<<grid, block, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace kda
