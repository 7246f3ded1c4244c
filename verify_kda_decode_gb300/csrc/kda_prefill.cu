// kda_prefill.cu -- chunked prefill of the KDA mixer step on the tcgen05 tensor cores.
//
// The prompt is cut into chunks of C = 64 tokens (KDA linear attention with a prefill path,
// Kimi K3 NVFP4 on Rubin page, section 3; chunked / WY form of the gated delta rule).  Within
// a chunk with entry state S0, per key channel the cumulative log-decay Gam_t (inclusive) and
// beta-scaled pseudo-values Ut = beta * u satisfy
//   (I + diag(beta) A) X = diag(beta) [Ktil | V],   A[t][s] = sum_c k_t[c] k_s[c] e^(Gam_t - Gam_s)[c]  (s < t)
//   X = [W | U]:   Ut = U - W S0,     Ktil_t = k_t e^(Gam_t)
//   O = Qtil S0 + Aqk Ut,              Qtil_t = q_t e^(Gam_t),  Aqk[t][s] = sum_c q_t k_s e^(Gam_t - Gam_s)  (s <= t)
//   S_end = Diag(e^(Gam_last)) S0 + Kbar^T Ut,   Kbar_s = k_s e^(Gam_last - Gam_s)
// Three launches:
//   prep  (one CTA per sequence x head x chunk, all chunks in parallel): short conv + SiLU,
//         q/k L2 norms, beta; the f_b projection W_fb[h] F_a^T as one tcgen05 MMA (bf16 inputs
//         are exact, f32 accumulation) -> log-decay and its running sum Gam; the gated Gram
//         blocks A and Aqk on tcgen05 in 16-token column blocks, each referenced to the middle
//         token of its block so that no factor exceeds e^(8 |log alpha|); X by forward
//         substitution in FP32; W, U, Qtil, Kbar^T, Aqk, e^(Gam_last) -> workspace.
//   scan  (one CTA per sequence x head x 32-column block of S, chunks in order): per chunk
//         [W; Qtil] S, then Ut = U - W S, then Kbar^T Ut and Aqk Ut on tcgen05, S update in
//         registers; pre-norm outputs -> workspace; final state and conv window -> slot.
//   norm  gated RMSNorm of the outputs.
// Every tensor-core product of FP32 operands runs as three bf16 MMAs (hi*hi + hi*lo + lo*hi,
// ~16 significant bits per operand) accumulating in FP32 tensor memory.
#include <cstddef>

#include "kda_prefill.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

constexpr int C = kPrefillChunk;                 // 64
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kMaxNegLogDecay = 10.0f;        // |log alpha| per token the Gram staging supports
constexpr int kScanCols = 32;                    // columns of S per scan CTA
// Per (sequence, head, chunk) workspace record, in floats.
constexpr int kOffW = 0, kOffU = C * 128, kOffQt = 2 * C * 128, kOffKbT = 3 * C * 128,
              kOffAqk = 4 * C * 128, kOffD = 4 * C * 128 + C * C, kChunkFloats = kOffD + 128;
static_assert((kChunkFloats * 4) % 256 == 0, "record alignment");

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float softplusf_(float x) { return x > 20.0f ? x : log1pf(expf(x)); }

template <int W>
__device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// All threads wait for a tensor-core commit; on a timeout the error is flagged and false is
// returned (the caller then frees its tensor memory and returns).
__device__ __forceinline__ bool wait_commit(uint64_t *bar, uint32_t parity, int *err)
{
    const bool ok = mbar_wait_bounded(bar, parity, kWaitLimitNs);
    if (__syncthreads_or(!ok)) {
        if (threadIdx.x == 0) {
            atomicOr(err, KDA_DEVERR_TIMEOUT);
            mbar_wait_bounded(bar, parity, kWaitLimitNs);
        }
        return false;
    }
    tc::fence_after_sync();
    return true;
}

// ============================================================================ prep

constexpr int NTA = 256;

struct PrepSmem {
    // phase 1: f_b operands; phase 2: Gram operands (same bytes)
    alignas(1024) uint8_t opnd[2 * 128 * 128 * 2 + 2 * 16 * 128 * 2];   // 72 KiB
    alignas(16) float q[C][128];
    alignas(16) float k[C][128];
    alignas(16) float v[C][128];
    alignas(16) float gam[C][128];
    alignas(16) float akk[C][C];
    alignas(16) float beta[C];
    alignas(8) uint64_t bar;
    uint32_t tmem;
};

__global__ void __launch_bounds__(NTA, 1) kda_chunk_prep(const RecurrentParams p, float *ws, int n_chunks)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    PrepSmem &sm = *reinterpret_cast<PrepSmem *>(smem_raw);
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int H = p.H, HC = H * kDk, L = p.T;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = c * C, n = L - t0 < C ? L - t0 : C;
    const int slot = __ldg(p.slot_ids + b);
    if (slot < 0 || slot >= p.num_slots) {
        if (tid == 0 && c == 0 && h == 0) atomicOr(p.err_word, KDA_DEVERR_SLOT);
        return;
    }
    float *rec = ws + ((size_t)(b * H + h) * n_chunks + c) * kChunkFloats;

    if (warp == 0) tc::tmem_alloc(&sm.tmem, 128);
    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        fence_mbar_init();
    }
    // f_b operands: W_fb rows of the head (A, 128 x 128) and f_a of the chunk (B, 64 x 128)
    uint8_t *wcm = sm.opnd, *facm = sm.opnd + 128 * 128 * 2;
    for (int qd = tid; qd < 128 * 16; qd += NTA) {
        int r, k;
        tc::cm_chunk(qd, 128, r, k);
        *reinterpret_cast<uint4 *>(wcm + qd * 16) = __ldg(reinterpret_cast<const uint4 *>(p.W_fb + ((size_t)h * kDk + r) * kRank + k));
    }
    for (int qd = tid; qd < C * 16; qd += NTA) {
        int r, k;
        tc::cm_chunk(qd, 128, r, k);
        uint4 val = make_uint4(0, 0, 0, 0);
        if (r < n) val = __ldg(reinterpret_cast<const uint4 *>(p.f_a + ((size_t)b * L + t0 + r) * kRank + k));
        *reinterpret_cast<uint4 *>(facm + qd * 16) = val;
    }
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = sm.tmem;
    uint32_t phase = 0;
    if (tid == 0) {
        tc::mma_tiles(tmem, smem_u32(wcm), 128, smem_u32(facm), 128, C, 0, 8, false);
        tc::commit(&sm.bar);
    }

    // ---- short causal conv + SiLU (window from the slot for chunk 0, else the 3 raw inputs
    //      before the chunk); padded tokens are zero
    for (int it = tid; it < 3 * kDk; it += NTA) {
        const int tens = it / kDk, cc = it % kDk, ch = h * kDk + cc;
        const __nv_bfloat16 *src = tens == 0 ? p.q : tens == 1 ? p.k : p.v;
        const uint2 wv = __ldg(reinterpret_cast<const uint2 *>(p.conv_w + ((size_t)tens * HC + ch) * kConv));
        const float w0 = __uint_as_float(wv.x << 16), w1 = __uint_as_float(wv.x & 0xffff0000u);
        const float w2 = __uint_as_float(wv.y << 16), w3 = __uint_as_float(wv.y & 0xffff0000u);
        float z[3];
        for (int j = 0; j < 3; j++) {
            const int tok = t0 - 3 + j;
            z[j] = tok >= 0 ? bf2f(src[((size_t)b * L + tok) * HC + ch])
                            : bf2f(p.conv_state[(((size_t)slot * 3 + tens) * kTaps + (tok + 3)) * HC + ch]);
        }
        float *dst = tens == 0 ? &sm.q[0][0] : tens == 1 ? &sm.k[0][0] : &sm.v[0][0];
        for (int t = 0; t < C; t++) {
            float y = 0.f;
            if (t < n) {
                const float x = bf2f(src[((size_t)b * L + t0 + t) * HC + ch]);
                float acc = w0 * z[0];
                acc = fmaf(w1, z[1], acc);
                acc = fmaf(w2, z[2], acc);
                acc = fmaf(w3, x, acc);
                y = acc / (1.0f + expf(-acc));
                z[0] = z[1];
                z[1] = z[2];
                z[2] = x;
            }
            dst[t * 128 + cc] = y;
        }
    }
    if (tid < C) sm.beta[tid] = tid < n ? sigmoidf_(bf2f(p.beta[((size_t)b * L + t0 + tid) * H + h])) : 0.f;
    __syncthreads();
    // ---- q, k L2 norms (q also scaled by dk^-1/2); rows 0..63 q, 64..127 k
    for (int row = warp; row < 2 * C; row += NTA / 32) {
        float *x = row < C ? &sm.q[row][0] : &sm.k[row - C][0];
        float4 a = *reinterpret_cast<float4 *>(x + lane * 4);
        const float ss = group_sum<32>(a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w);
        const float f = (row < C ? rsqrtf((float)kDk) : 1.0f) / sqrtf(ss + p.l2_eps);
        a.x *= f; a.y *= f; a.z *= f; a.w *= f;
        *reinterpret_cast<float4 *>(x + lane * 4) = a;
    }
    // ---- decay: TMEM holds graw[i = lane row][t = column]
    bool ok = wait_commit(&sm.bar, phase, p.err_word);
    phase ^= 1;
    if (ok && warp < 4) {
        const int i = warp * 32 + lane;
        float g0[32], g1[32];
        tc::ld32(tc::taddr(tmem, warp * 32, 0), g0);
        tc::ld32(tc::taddr(tmem, warp * 32, 32), g1);
        const float a = expf(__ldg(p.A_log + h)), db = __ldg(p.dt_bias + h * kDk + i);
        float G = 0.f;
        bool range_ok = true;
        for (int t = 0; t < C; t++) {
            const float gr = t < 32 ? g0[t] : g1[t - 32];
            float g = 0.f;
            if (t < n) g = -a * softplusf_(gr + db);
            range_ok &= g >= -kMaxNegLogDecay;
            G += g;
            sm.gam[t][i] = G;
        }
        if (!range_ok) atomicOr(p.err_word, KDA_DEVERR_DECAY);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---- gated Gram blocks: column block J (tokens 16J..16J+15), reference token m = 16J + 7
    uint8_t *ahi = sm.opnd, *alo = ahi + 128 * 128 * 2, *bhi = alo + 128 * 128 * 2, *blo = bhi + 16 * 128 * 2;
    for (int J = 0; J < 4 && ok; J++) {
        const int m = 16 * J + 7;
        for (int qd = tid; qd < 128 * 16; qd += NTA) {
            int r, k;
            tc::cm_chunk(qd, 128, r, k);
            const int t = r & (C - 1);
            const float *src = r < C ? &sm.k[t][k] : &sm.q[t][k];
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; e++)
                x[e] = t < 16 * J ? 0.f : src[e] * __expf(sm.gam[t][k + e] - sm.gam[m][k + e]);
            uint4 hi, lo;
            tc::split8(x, hi, lo);
            *reinterpret_cast<uint4 *>(ahi + qd * 16) = hi;
            *reinterpret_cast<uint4 *>(alo + qd * 16) = lo;
        }
        for (int qd = tid; qd < 16 * 16; qd += NTA) {
            int r, k;
            tc::cm_chunk(qd, 128, r, k);
            const int j = 16 * J + r;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; e++) x[e] = sm.k[j][k + e] * __expf(sm.gam[m][k + e] - sm.gam[j][k + e]);
            uint4 hi, lo;
            tc::split8(x, hi, lo);
            *reinterpret_cast<uint4 *>(bhi + qd * 16) = hi;
            *reinterpret_cast<uint4 *>(blo + qd * 16) = lo;
        }
        tc::fence_smem_to_async();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (tid == 0) {
            tc::mma_split3(tmem + 64 + 16 * J, smem_u32(ahi), smem_u32(alo), 128, smem_u32(bhi), smem_u32(blo), 128, 16, 8, false);
            tc::commit(&sm.bar);
        }
        ok = wait_commit(&sm.bar, phase, p.err_word);
        phase ^= 1;
    }
    if (ok) {
        // lanes 0..63: A[i][j] (kept for j < i); lanes 64..127: Aqk[i][j] (kept for j <= i)
        const int wq = warp & 3, half = warp >> 2;
        float g[32];
        tc::ld32(tc::taddr(tmem, 32 * wq, 64 + 32 * half), g);
        const int row = 32 * wq + lane;
        for (int jj = 0; jj < 32; jj++) {
            const int j = 32 * half + jj;
            if (row < C) sm.akk[row][j] = j < row ? g[jj] : 0.f;
            else rec[kOffAqk + (row - C) * C + j] = j <= row - C ? g[jj] : 0.f;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 128);
    if (!ok) return;

    // ---- forward substitution, one column per thread: columns 0..127 Ktil, 128..255 V
    {
        const int col = tid;
        float x[C];
#pragma unroll
        for (int t = 0; t < C; t++) {
            float rhs = col < 128 ? sm.k[t][col] * __expf(sm.gam[t][col]) : sm.v[t][col - 128];
#pragma unroll
            for (int s = 0; s < t; s++) rhs = fmaf(-sm.akk[t][s], x[s], rhs);
            x[t] = sm.beta[t] * rhs;
        }
        float *dst = rec + (col < 128 ? kOffW + col : kOffU + col - 128);
#pragma unroll
        for (int t = 0; t < C; t++) dst[t * 128] = x[t];
    }
    // ---- Qtil, Kbar^T (dk-major), e^(Gam_last)
    for (int idx = tid; idx < C * 128; idx += NTA) {
        const int t = idx >> 7, i = idx & 127;
        rec[kOffQt + idx] = sm.q[t][i] * __expf(sm.gam[t][i]);
    }
    if (tid < 128) {
        const int i = tid;
        const float gl = sm.gam[C - 1][i];   // padded tokens keep Gam constant
        for (int t = 0; t < C; t += 4) {
            float4 o;
            o.x = sm.k[t][i] * __expf(gl - sm.gam[t][i]);
            o.y = sm.k[t + 1][i] * __expf(gl - sm.gam[t + 1][i]);
            o.z = sm.k[t + 2][i] * __expf(gl - sm.gam[t + 2][i]);
            o.w = sm.k[t + 3][i] * __expf(gl - sm.gam[t + 3][i]);
            *reinterpret_cast<float4 *>(rec + kOffKbT + i * C + t) = o;
        }
        rec[kOffD + i] = __expf(gl);
    }
}

// ============================================================================ scan

constexpr int NTB = 128;

struct ScanSmem {
    alignas(1024) uint8_t a1[2][128 * 128 * 2];   // [W; Qtil] hi / lo, K = dk
    alignas(1024) uint8_t b1[2][kScanCols * 128 * 2];   // S^T hi / lo, K = dk
    alignas(1024) uint8_t a2[2][128 * C * 2];     // Kbar^T hi / lo, K = tokens
    alignas(1024) uint8_t a3[2][128 * C * 2];     // [0; Aqk] hi / lo, K = tokens
    alignas(1024) uint8_t b2[2][kScanCols * C * 2];   // Ut^T hi / lo, K = tokens
    alignas(8) uint64_t bar;
    uint32_t tmem;
};

template <typename ST>
__global__ void __launch_bounds__(NTB, 1) kda_chunk_scan(const RecurrentParams p, const float *ws, float *o_pre, int n_chunks)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    ScanSmem &sm = *reinterpret_cast<ScanSmem *>(smem_raw);
    const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int H = p.H, HC = H * kDk, L = p.T;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int slot = __ldg(p.slot_ids + b);
    if (slot < 0 || slot >= p.num_slots) return;   // flagged by the prep launch
    const int col0 = blk * kScanCols;

    // S rows i = tid, columns col0 .. col0 + 31, FP32 in registers
    ST *tile = reinterpret_cast<ST *>(p.state) + ((size_t)slot * H + h) * (kDk * kDv);
    float S[kScanCols];
#pragma unroll
    for (int j = 0; j < kScanCols; j++) S[j] = (float)tile[(size_t)tid * kDv + col0 + j];

    if (warp == 0) tc::tmem_alloc(&sm.tmem, 64);
    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        fence_mbar_init();
    }
    // rows 0..63 of [0; Aqk] stay zero
    for (int qd = tid; qd < 64 * (C / 8); qd += NTB) {
        *reinterpret_cast<uint4 *>(sm.a3[0] + qd * 16) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(sm.a3[1] + qd * 16) = make_uint4(0, 0, 0, 0);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = sm.tmem, d1 = tmem, d2 = tmem + 32;
    uint32_t phase = 0;
    bool ok = true;

    for (int c = 0; c < n_chunks && ok; c++) {
        const int t0 = c * C, n = L - t0 < C ? L - t0 : C;
        const float *rec = ws + ((size_t)(b * H + h) * n_chunks + c) * kChunkFloats;
        // [W; Qtil] (128 x 128), Kbar^T (128 x 64), Aqk rows of [0; Aqk]
        for (int qd = tid; qd < 128 * 16; qd += NTB) {
            int r, k;
            tc::cm_chunk(qd, 128, r, k);
            const float *src = rec + (r < C ? kOffW + r * 128 : kOffQt + (r - C) * 128) + k;
            float x[8];
            *reinterpret_cast<float4 *>(x) = *reinterpret_cast<const float4 *>(src);
            *reinterpret_cast<float4 *>(x + 4) = *reinterpret_cast<const float4 *>(src + 4);
            uint4 hi, lo;
            tc::split8(x, hi, lo);
            *reinterpret_cast<uint4 *>(sm.a1[0] + qd * 16) = hi;
            *reinterpret_cast<uint4 *>(sm.a1[1] + qd * 16) = lo;
        }
        for (int qd = tid; qd < 128 * (C / 8); qd += NTB) {
            int r, k;
            tc::cm_chunk(qd, C, r, k);
            const float *src = rec + kOffKbT + r * C + k;
            float x[8];
            *reinterpret_cast<float4 *>(x) = *reinterpret_cast<const float4 *>(src);
            *reinterpret_cast<float4 *>(x + 4) = *reinterpret_cast<const float4 *>(src + 4);
            uint4 hi, lo;
            tc::split8(x, hi, lo);
            *reinterpret_cast<uint4 *>(sm.a2[0] + qd * 16) = hi;
            *reinterpret_cast<uint4 *>(sm.a2[1] + qd * 16) = lo;
            if (r >= 64) {   // the same chunk position of [0; Aqk]
                const float *sq = rec + kOffAqk + (r - 64) * C + k;
                *reinterpret_cast<float4 *>(x) = *reinterpret_cast<const float4 *>(sq);
                *reinterpret_cast<float4 *>(x + 4) = *reinterpret_cast<const float4 *>(sq + 4);
                tc::split8(x, hi, lo);
                *reinterpret_cast<uint4 *>(sm.a3[0] + qd * 16) = hi;
                *reinterpret_cast<uint4 *>(sm.a3[1] + qd * 16) = lo;
            }
        }
        // S^T (32 x 128): element (n = column j, k = row i)
#pragma unroll
        for (int j = 0; j < kScanCols; j++) {
            __nv_bfloat16 hi, lo;
            tc::split_bf16(S[j], hi, lo);
            const uint32_t off = tc::cm_off(j, tid, 128);
            *reinterpret_cast<__nv_bfloat16 *>(sm.b1[0] + off) = hi;
            *reinterpret_cast<__nv_bfloat16 *>(sm.b1[1] + off) = lo;
        }
        tc::fence_smem_to_async();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (tid == 0) {
            tc::mma_split3(d1, smem_u32(sm.a1[0]), smem_u32(sm.a1[1]), 128, smem_u32(sm.b1[0]), smem_u32(sm.b1[1]), 128, kScanCols, 8, false);
            tc::commit(&sm.bar);
        }
        ok = wait_commit(&sm.bar, phase, p.err_word);
        phase ^= 1;
        if (!ok) break;
        // Ut = U - W S for token t = tid (< 64), stored transposed as the B operand (32 x 64)
        if (warp < 2) {
            float wsv[32];
            tc::ld32(tc::taddr(tmem, 32 * warp, 0), wsv);
            const int t = tid;
            const float *u = rec + kOffU + t * 128 + col0;
#pragma unroll
            for (int j = 0; j < kScanCols; j++) {
                const float ut = t < n ? u[j] - wsv[j] : 0.f;
                __nv_bfloat16 hi, lo;
                tc::split_bf16(ut, hi, lo);
                const uint32_t off = tc::cm_off(j, t, C);
                *reinterpret_cast<__nv_bfloat16 *>(sm.b2[0] + off) = hi;
                *reinterpret_cast<__nv_bfloat16 *>(sm.b2[1] + off) = lo;
            }
        }
        tc::fence_smem_to_async();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (tid == 0) {
            // Kbar^T Ut -> d2;  [0; Aqk] Ut accumulated onto [W S; Qtil S] -> rows 64.. = O
            tc::mma_split3(d2, smem_u32(sm.a2[0]), smem_u32(sm.a2[1]), C, smem_u32(sm.b2[0]), smem_u32(sm.b2[1]), C, kScanCols, 4, false);
            tc::mma_split3(d1, smem_u32(sm.a3[0]), smem_u32(sm.a3[1]), C, smem_u32(sm.b2[0]), smem_u32(sm.b2[1]), C, kScanCols, 4, true);
            tc::commit(&sm.bar);
        }
        ok = wait_commit(&sm.bar, phase, p.err_word);
        phase ^= 1;
        if (!ok) break;
        {
            float ds[32];
            tc::ld32(tc::taddr(tmem, 32 * warp, 32), ds);
            const float dcay = rec[kOffD + tid];
#pragma unroll
            for (int j = 0; j < kScanCols; j++) S[j] = fmaf(dcay, S[j], ds[j]);
        }
        if (warp >= 2) {
            float o[32];
            tc::ld32(tc::taddr(tmem, 32 * warp, 0), o);
            const int t = tid - 64;
            if (t < n) {
                float *dst = o_pre + (((size_t)b * L + t0 + t) * H + h) * kDv + col0;
#pragma unroll
                for (int j = 0; j < kScanCols; j += 4)
                    *reinterpret_cast<float4 *>(dst + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
            }
        }
        tc::fence_before_sync();
        __syncthreads();   // the operands of this chunk are no longer read
        tc::fence_after_sync();
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 64);
    if (!ok) return;
    // final state (one rounding to the storage dtype)
#pragma unroll
    for (int j = 0; j < kScanCols; j++) tile[(size_t)tid * kDv + col0 + j] = (ST)S[j];
    // final conv window of the head's channels: z = [window, x_0 .. x_{L-1}], keep z[L .. L+2]
    if (blk == 0) {
        for (int it = tid; it < 3 * kDk; it += NTB) {
            const int tens = it / kDk, ch = h * kDk + it % kDk;
            const __nv_bfloat16 *src = tens == 0 ? p.q : tens == 1 ? p.k : p.v;
            __nv_bfloat16 w[3];
            for (int j = 0; j < 3; j++) {
                const int zi = L + j;   // index into z
                w[j] = zi < 3 ? p.conv_state[(((size_t)slot * 3 + tens) * kTaps + zi) * HC + ch]
                              : src[((size_t)b * L + zi - 3) * HC + ch];
            }
            for (int j = 0; j < 3; j++) p.conv_state[(((size_t)slot * 3 + tens) * kTaps + j) * HC + ch] = w[j];
        }
    }
}

// ============================================================================ norm

__global__ void __launch_bounds__(256) kda_chunk_norm(const RecurrentParams p, const float *o_pre)
{
    const long wid = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long n_rows = (long)p.B * p.T * p.H;
    if (wid >= n_rows) return;
    const int h = (int)(wid % p.H);
    const float4 o = *reinterpret_cast<const float4 *>(o_pre + wid * kDv + lane * 4);
    const float ss = group_sum<32>(o.x * o.x + o.y * o.y + o.z * o.z + o.w * o.w);
    const float r = rsqrtf(ss * (1.0f / kDv) + p.norm_eps);
    const size_t base = (size_t)(wid / p.H) * (size_t)(p.H * kDv) + (size_t)h * kDv + lane * 4;
    const float ov[4] = {o.x, o.y, o.z, o.w};
    __nv_bfloat16 y[4];
#pragma unroll
    for (int e = 0; e < 4; e++)
        y[e] = __float2bfloat16_rn(ov[e] * r * __ldg(p.norm_w + lane * 4 + e) * sigmoidf_(bf2f(p.gate[base + e])));
    *reinterpret_cast<uint2 *>(p.out + base) = make_uint2(tc::pack2(y[0], y[1]), tc::pack2(y[2], y[3]));
}

template <typename F>
cudaError_t set_smem(F kern, size_t bytes, int &configured)
{
    if (configured >= (int)bytes) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) configured = (int)bytes;
    return e;
}

}  // namespace

size_t prefill_workspace_bytes(int H, int B, int L)
{
    if (H <= 0 || B <= 0 || L <= 0) return 0;
    const size_t n_chunks = (size_t)(L + C - 1) / C;
    return (size_t)B * H * n_chunks * kChunkFloats * sizeof(float) + (size_t)B * L * H * kDv * sizeof(float);
}

cudaError_t launch_prefill(const RecurrentParams &p, bool bf16_state, void *workspace, cudaStream_t stream)
{
    static int cfg_prep = 0, cfg_scan_f = 0, cfg_scan_b = 0;
    const int n_chunks = (p.T + C - 1) / C;
    float *ws = static_cast<float *>(workspace);
    float *o_pre = ws + (size_t)p.B * p.H * n_chunks * kChunkFloats;
    cudaError_t e = set_smem(kda_chunk_prep, sizeof(PrepSmem), cfg_prep);
    if (e != cudaSuccess) return e;
    kda_chunk_prep<<<dim3((unsigned)n_chunks, (unsigned)p.H, (unsigned)p.B), NTA, sizeof(PrepSmem), stream>>>(p, ws, n_chunks);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const dim3 sgrid(kDv / kScanCols, (unsigned)p.H, (unsigned)p.B);
    if (bf16_state) {
        if ((e = set_smem(kda_chunk_scan<__nv_bfloat16>, sizeof(ScanSmem), cfg_scan_b)) != cudaSuccess) return e;
        kda_chunk_scan<__nv_bfloat16><<<sgrid, NTB, sizeof(ScanSmem), stream>>>(p, ws, o_pre, n_chunks);
    } else {
        if ((e = set_smem(kda_chunk_scan<float>, sizeof(ScanSmem), cfg_scan_f)) != cudaSuccess) return e;
        kda_chunk_scan<float><<<sgrid, NTB, sizeof(ScanSmem), stream>>>(p, ws, o_pre, n_chunks);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const long rows = (long)p.B * p.T * p.H;
    kda_chunk_norm<<<(unsigned)((rows * 32 + 255) / 256), 256, 0, stream>>>(p, o_pre);
    return cudaGetLastError();
}

}  // namespace kda
