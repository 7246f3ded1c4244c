// kda_decode.cu -- single-token decode and multi-token draft verify of the KDA mixer step as a
// persistent, software-pipelined kernel.
//
// Work item = one (sequence, head) tile: the 128 x 128 recurrent state of that head in the
// sequence's slot.  Each CTA (256 threads) walks the items i = blockIdx.x + j * gridDim.x.  The
// state tiles are staged through shared memory by 1-D bulk async copies (TMA) into NSTAGE
// stages, each guarded by an mbarrier: while item j is computed, the tiles of items j+1..
// are already streaming in, so HBM sees a continuous read stream; updated tiles (decode) or
// FP32 draft records (verify) leave the registers with coalesced 128-bit stores.
//
// Per item the CTA fuses ("KDA fuses the f_b projection, convolution, FP32 recurrence and gated
// output normalization", NVFP4 Kimi K3 targets page, Description), for all T tokens at once:
//   f_b projection W_fb[h] . f_a (16 lanes per W row, shuffle-reduced) -> alpha = exp(g);
//   short causal conv + SiLU of the head's q, k, v channels (window in registers);
//   |q|^2, |k|^2, q.k per token (warp reductions) and beta;
// then, token by token, on the FP32 register tile:
//   S <- Diag(alpha) S with S^T k and S^T q in the same sweep (cross-warp reduction in smem),
//   u = v - S^T k, o = S^T q + beta u (k.q), gated RMSNorm of o, S += beta k u^T.
// Verify writes the FP32 state and the conv window after every draft token and leaves the
// slot untouched ("FP32 per-token draft records with either SSM storage dtype", same page;
// per-token KDA verify states, Kimi K3 on modeling_v2 page, section 5); decode writes the
// state, rounded once to the storage dtype, and the window back to the slot.
#include "kda_decode.cuh"
#include "kda_ptx.cuh"

namespace kda {
namespace {

constexpr int NT = 256;
constexpr int NSTAGE = 2;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: no wait of this kernel can spin longer

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
    static constexpr int BYTES = kDk * kDv * sizeof(ST);
};

__device__ __forceinline__ void unpack(const uint4 &r, float *f, float)
{
    f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
}

__device__ __forceinline__ void unpack(const uint4 &r, float *f, __nv_bfloat16)
{
    f[0] = bf16_lo(r.x); f[1] = bf16_hi(r.x); f[2] = bf16_lo(r.y); f[3] = bf16_hi(r.y);
    f[4] = bf16_lo(r.z); f[5] = bf16_hi(r.z); f[6] = bf16_lo(r.w); f[7] = bf16_hi(r.w);
}

__device__ __forceinline__ uint4 pack(const float *f, float)
{
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
}

__device__ __forceinline__ uint4 pack(const float *f, __nv_bfloat16)
{
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

// Fixed part of the shared memory (after the stages); the per-token gate arrays follow it.
struct __align__(16) Fixed {
    uint64_t full[NSTAGE];
    float red[NT / 32][2][kDv];   // per-warp partial S^T k / S^T q
    float u[kDv];
    float rms[4];
    int flag;
};

// Per-token gate arrays, T rows each: alpha (also f_b accumulator), q, k, v (post conv, raw),
// f_a (input), norms (|q|^2, |k|^2, q.k, beta).
struct GateArrays {
    float *alpha, *q, *k, *v, *fa, *nrm;
};

__host__ __device__ constexpr size_t gate_bytes(int T) { return (size_t)T * (5 * 128 + 4) * sizeof(float); }

template <typename ST>
__host__ __device__ constexpr size_t stage_bytes() { return (size_t)NSTAGE * Tile<ST>::BYTES; }

template <typename ST>
size_t smem_bytes(int T) { return stage_bytes<ST>() + sizeof(Fixed) + gate_bytes(T); }

struct ConvItem {
    int tensor, ch;
    float w[kConv];
    __nv_bfloat16 win[kTaps];
};

// Gate phase of one item for its T tokens; ends with __syncthreads().
template <bool RECORDS>
__device__ __forceinline__ void gate_phase(const RecurrentParams &p, const GateArrays &g, int b,
                                           int h, int slot)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, H = p.H, HC = H * kDk, T = p.T;
    const size_t tok0 = (size_t)b * T;
    // f_a of the T tokens -> smem; conv items -> registers (and their inputs)
    for (int i = tid; i < T * kRank; i += NT) g.fa[i] = bf2f(p.f_a[tok0 * kRank + i]);
    ConvItem cv[2];
    const int n_items = tid < kDv ? 2 : 1;
#pragma unroll
    for (int it = 0; it < 2; it++) {
        if (it < n_items) {
            cv[it].tensor = it == 0 ? (tid < kDk ? 0 : 1) : 2;
            cv[it].ch = h * kDk + (tid & (kDk - 1));
            const uint2 w = __ldg(reinterpret_cast<const uint2 *>(p.conv_w + ((size_t)cv[it].tensor * HC + cv[it].ch) * kConv));
            cv[it].w[0] = bf16_lo(w.x); cv[it].w[1] = bf16_hi(w.x);
            cv[it].w[2] = bf16_lo(w.y); cv[it].w[3] = bf16_hi(w.y);
#pragma unroll
            for (int j = 0; j < kTaps; j++)
                cv[it].win[j] = p.conv_state[(((size_t)slot * 3 + cv[it].tensor) * kTaps + j) * HC + cv[it].ch];
        }
    }
    __syncthreads();   // fa visible
    // a1: graw[t][i] = W_fb[h*128+i] . f_a[t]; half-warp hw owns rows hw + 16 m, lane li owns r in [8li, 8li+8)
    {
        const int hw = tid >> 4, li = tid & 15;
#pragma unroll 2
        for (int m = 0; m < 8; m++) {
            const int i = hw + 16 * m;
            const uint4 wr = __ldg(reinterpret_cast<const uint4 *>(p.W_fb + ((size_t)h * kDk + i) * kRank + li * 8));
            const float w0 = bf16_lo(wr.x), w1 = bf16_hi(wr.x), w2 = bf16_lo(wr.y), w3 = bf16_hi(wr.y);
            const float w4 = bf16_lo(wr.z), w5 = bf16_hi(wr.z), w6 = bf16_lo(wr.w), w7 = bf16_hi(wr.w);
            for (int t = 0; t < T; t++) {
                const float4 f0 = *reinterpret_cast<const float4 *>(g.fa + t * kRank + li * 8);
                const float4 f1 = *reinterpret_cast<const float4 *>(g.fa + t * kRank + li * 8 + 4);
                float acc = w0 * f0.x;
                acc = fmaf(w1, f0.y, acc);
                acc = fmaf(w2, f0.z, acc);
                acc = fmaf(w3, f0.w, acc);
                acc = fmaf(w4, f1.x, acc);
                acc = fmaf(w5, f1.y, acc);
                acc = fmaf(w6, f1.z, acc);
                acc = fmaf(w7, f1.w, acc);
                acc = group_sum<16>(acc);
                if (li == m) g.alpha[t * kDk + i] = acc;
            }
        }
    }
    // a4: conv + SiLU per token, window shift; verify records the window after each token
#pragma unroll
    for (int it = 0; it < 2; it++) {
        if (it < n_items) {
            const int tens = cv[it].tensor, ch = cv[it].ch, c = ch - h * kDk;
            const __nv_bfloat16 *src = tens == 0 ? p.q : (tens == 1 ? p.k : p.v);
            float *dst = tens == 0 ? g.q : (tens == 1 ? g.k : g.v);
            for (int t = 0; t < T; t++) {
                const __nv_bfloat16 x = src[(tok0 + t) * HC + ch];
                float acc = cv[it].w[0] * bf2f(cv[it].win[0]);
                acc = fmaf(cv[it].w[1], bf2f(cv[it].win[1]), acc);
                acc = fmaf(cv[it].w[2], bf2f(cv[it].win[2]), acc);
                acc = fmaf(cv[it].w[3], bf2f(x), acc);
                dst[t * kDk + c] = acc / (1.0f + expf(-acc));
                cv[it].win[0] = cv[it].win[1];
                cv[it].win[1] = cv[it].win[2];
                cv[it].win[2] = x;
                if (RECORDS) {
#pragma unroll
                    for (int j = 0; j < kTaps; j++)
                        p.rec_conv[(((tok0 + t) * 3 + tens) * kTaps + j) * HC + ch] = cv[it].win[j];
                }
            }
            if (!RECORDS) {
#pragma unroll
                for (int j = 0; j < kTaps; j++)
                    p.conv_state[(((size_t)slot * 3 + tens) * kTaps + j) * HC + ch] = cv[it].win[j];
            }
        }
    }
    __syncthreads();   // graw, q, k, v visible
    // a2: decay; a5: |q|^2, |k|^2, q.k; a3: beta
    const float a_h = expf(p.A_log[h]);
    for (int i = tid; i < T * kDk; i += NT) {
        const int c = i & (kDk - 1);
        g.alpha[i] = expf(-a_h * softplusf_(g.alpha[i] + p.dt_bias[h * kDk + c]));
    }
    for (int pr = warp; pr < 3 * T; pr += NT / 32) {
        const int t = pr / 3, kind = pr % 3;
        const float *a = (kind == 1 ? g.k : g.q) + t * kDk;
        const float *c = (kind == 0 ? g.q : g.k) + t * kDk;
        const float4 x = *reinterpret_cast<const float4 *>(a + lane * 4);
        const float4 y = *reinterpret_cast<const float4 *>(c + lane * 4);
        float s = x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
        s = group_sum<32>(s);
        if (lane == 0) g.nrm[t * 4 + kind] = s;
    }
    for (int t = tid; t < T; t += NT) g.nrm[t * 4 + 3] = sigmoidf_(bf2f(p.beta[(tok0 + t) * H + h]));
    __syncthreads();
}

template <typename ST, bool RECORDS>
__global__ void __launch_bounds__(NT, 1) kda_stream_kernel(const RecurrentParams p)
{
    using TL = Tile<ST>;
    constexpr int VEC = TL::VEC, TPR = TL::TPR, RPP = TL::RPP, NP = TL::NP;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *stages = smem;
    Fixed &fx = *reinterpret_cast<Fixed *>(smem + stage_bytes<ST>());
    float *gbase = reinterpret_cast<float *>(smem + stage_bytes<ST>() + sizeof(Fixed));
    const int T = p.T, H = p.H;
    GateArrays g;
    g.alpha = gbase;
    g.q = g.alpha + T * kDk;
    g.k = g.q + T * kDk;
    g.v = g.k + T * kDk;
    g.fa = g.v + T * kDv;
    g.nrm = g.fa + T * kRank;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_items = p.B * H;
    const int col = (tid % TPR) * VEC, row0 = tid / TPR;
    const float q_scale = rsqrtf((float)kDk);

    auto item_slot = [&](int it) -> int { return p.slot_ids[it / H]; };
    auto valid_slot = [&](int s) -> bool { return s >= 0 && s < p.num_slots; };
    // thread 0 only: start the copy of item `it` into stage `s` (skipped for a bad slot)
    auto issue = [&](int it, int s) {
        if (it >= n_items) return;
        const int slot = item_slot(it);
        if (!valid_slot(slot)) return;
        const ST *src = reinterpret_cast<const ST *>(p.state) + ((size_t)slot * H + (it % H)) * (kDk * kDv);
        mbar_arrive_expect_tx(&fx.full[s], TL::BYTES);
        bulk_load(stages + (size_t)s * TL::BYTES, src, TL::BYTES, &fx.full[s]);
    };

    if (tid == 0) {
        for (int s = 0; s < NSTAGE; s++) mbar_init(&fx.full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0)
        for (int s = 0; s < NSTAGE; s++) issue(blockIdx.x + s * gridDim.x, s);

    uint32_t phase = 0;   // bit s: parity of the next completion of stage s
    for (int j = 0;; j++) {
        const int it = blockIdx.x + j * gridDim.x;
        if (it >= n_items) break;
        const int s = j % NSTAGE, b = it / H, h = it % H, slot = item_slot(it);
        if (j > 0) __syncthreads();   // previous item's readers of the gate arrays are done
        if (!valid_slot(slot)) {
            if (tid == 0) {
                atomicOr(p.err_word, KDA_DEVERR_SLOT);
                issue(it + NSTAGE * gridDim.x, s);   // the stage stays free: refill it
            }
            continue;
        }
        gate_phase<RECORDS>(p, g, b, h, slot);

        // wait for the tile; a wait that runs out flags the error and ends the CTA
        const bool ok = mbar_wait_bounded(&fx.full[s], (phase >> s) & 1u, kWaitLimitNs);
        phase ^= 1u << s;
        if (__syncthreads_or(!ok)) {
            if (tid == 0) atomicOr(p.err_word, KDA_DEVERR_TIMEOUT);
            // drain the other stage's copy (bounded) so that no copy lands after exit
            for (int o = 1; o < NSTAGE; o++) {
                const int so = (s + o) % NSTAGE, ito = it + o * gridDim.x;
                if (ito < n_items && valid_slot(item_slot(ito)))
                    mbar_wait_bounded(&fx.full[so], (phase >> so) & 1u, kWaitLimitNs);
            }
            return;
        }
        float st[NP][VEC];
        {
            const ST *tile = reinterpret_cast<const ST *>(stages + (size_t)s * TL::BYTES);
#pragma unroll
            for (int pp = 0; pp < NP; pp++) {
                const uint4 r = *reinterpret_cast<const uint4 *>(tile + (size_t)(row0 + RPP * pp) * kDv + col);
                unpack(r, st[pp], ST());
            }
        }

        for (int t = 0; t < T; t++) {
            const size_t tok = (size_t)b * T + t;
            const float *nrm = g.nrm + t * 4;
            const float rq = q_scale / sqrtf(nrm[0] + p.l2_eps);
            const float rk = 1.0f / sqrtf(nrm[1] + p.l2_eps);
            const float kq = nrm[2] * rq * rk;
            const float beta = nrm[3];
            const float *al = g.alpha + t * kDk, *kv = g.k + t * kDk, *qv = g.q + t * kDk;

            // a6: decay + S^T k, S^T q
            float ak[VEC], aq[VEC];
#pragma unroll
            for (int c = 0; c < VEC; c++) ak[c] = aq[c] = 0.f;
#pragma unroll
            for (int pp = 0; pp < NP; pp++) {
                const int i = row0 + RPP * pp;
                const float a = al[i], kk = kv[i] * rk, qq = qv[i] * rq;
#pragma unroll
                for (int c = 0; c < VEC; c++) {
                    st[pp][c] *= a;
                    ak[c] = fmaf(st[pp][c], kk, ak[c]);
                    aq[c] = fmaf(st[pp][c], qq, aq[c]);
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
                    *reinterpret_cast<float4 *>(&fx.red[warp][0][col + c]) = make_float4(ak[c], ak[c + 1], ak[c + 2], ak[c + 3]);
                    *reinterpret_cast<float4 *>(&fx.red[warp][1][col + c]) = make_float4(aq[c], aq[c + 1], aq[c + 2], aq[c + 3]);
                }
            }
            __syncthreads();
            // the stage has been read into registers: start the copy of item j + NSTAGE into it
            if (t == 0 && tid == 0) issue(it + NSTAGE * gridDim.x, s);

            // u, o, RMS partials
            float o = 0.f;
            if (tid < kDv) {
                float stk = 0.f, stq = 0.f;
#pragma unroll
                for (int w = 0; w < NT / 32; w++) { stk += fx.red[w][0][tid]; stq += fx.red[w][1][tid]; }
                const float u = g.v[t * kDv + tid] - stk;
                o = stq + beta * u * kq;
                fx.u[tid] = u;
                const float ss = group_sum<32>(o * o);
                if (lane == 0) fx.rms[warp] = ss;
            }
            __syncthreads();
            if (tid < kDv) {
                const float ms = (fx.rms[0] + fx.rms[1] + fx.rms[2] + fx.rms[3]) * (1.0f / kDv);
                const size_t oi = tok * (size_t)(H * kDv) + (size_t)h * kDv + tid;
                const float y = o * rsqrtf(ms + p.norm_eps) * __ldg(p.norm_w + tid) * sigmoidf_(bf2f(p.gate[oi]));
                p.out[oi] = __float2bfloat16_rn(y);
            }
            // S += beta k u^T
            float uu[VEC];
#pragma unroll
            for (int c = 0; c < VEC; c += 4) {
                const float4 u4 = *reinterpret_cast<const float4 *>(&fx.u[col + c]);
                uu[c] = u4.x; uu[c + 1] = u4.y; uu[c + 2] = u4.z; uu[c + 3] = u4.w;
            }
            float *rec = RECORDS ? p.rec_state + (tok * H + h) * (size_t)(kDk * kDv) : nullptr;
#pragma unroll
            for (int pp = 0; pp < NP; pp++) {
                const int i = row0 + RPP * pp;
                const float bk = beta * kv[i] * rk;
#pragma unroll
                for (int c = 0; c < VEC; c++) st[pp][c] = fmaf(bk, uu[c], st[pp][c]);
                if (RECORDS) {
#pragma unroll
                    for (int c = 0; c < VEC; c += 4)
                        __stcs(reinterpret_cast<float4 *>(rec + (size_t)i * kDv + col + c),
                               make_float4(st[pp][c], st[pp][c + 1], st[pp][c + 2], st[pp][c + 3]));
                }
            }
            if (t + 1 < T) __syncthreads();   // fx.u / fx.rms readers done before the next token
        }
        if (!RECORDS) {
            ST *tile = reinterpret_cast<ST *>(p.state) + ((size_t)slot * H + h) * (kDk * kDv);
#pragma unroll
            for (int pp = 0; pp < NP; pp++)
                __stcs(reinterpret_cast<uint4 *>(tile + (size_t)(row0 + RPP * pp) * kDv + col), pack(st[pp], ST()));
        }
    }
}

template <typename ST, bool RECORDS>
cudaError_t launch_one(const RecurrentParams &p, cudaStream_t stream)
{
    const size_t smem = smem_bytes<ST>(p.T);
    static int configured_smem = 0;
    static int sms = 0;
    if (configured_smem < (int)smem) {
        cudaError_t e = cudaFuncSetAttribute(kda_stream_kernel<ST, RECORDS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured_smem = (int)smem;
    }
    if (sms == 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_stream_kernel<ST, RECORDS>, NT, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const long items = (long)p.B * p.H;
    const int grid = (int)(items < (long)sms * per_sm ? items : (long)sms * per_sm);
    kda_stream_kernel<ST, RECORDS><<<grid, NT, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_stream(const RecurrentParams &p, bool bf16_state, bool records, cudaStream_t stream)
{
    if (bf16_state) return records ? launch_one<__nv_bfloat16, true>(p, stream) : launch_one<__nv_bfloat16, false>(p, stream);
    return records ? launch_one<float, true>(p, stream) : launch_one<float, false>(p, stream);
}

size_t stream_smem_bytes(bool bf16_state, int T)
{
    return bf16_state ? smem_bytes<__nv_bfloat16>(T) : smem_bytes<float>(T);
}

}  // namespace kda
