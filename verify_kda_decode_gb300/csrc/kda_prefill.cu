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
// Two launches:
//   prep  (one CTA of 16 warps per sequence x head x chunk, all chunks in parallel): short conv
//         + SiLU from rows staged by cp.async, q/k L2 norms, beta; the f_b projection
//         W_fb[h] F_a^T as one tcgen05 MMA (bf16 inputs are exact, f32 accumulation) ->
//         log-decay and its running sum Gam; the gated Gram matrices A and Aqk on tcgen05, with
//         one reference token for the whole chunk when the decay allows it; otherwise, for any
//         decay, the blocks below the diagonal referenced to the key block's last token (both
//         factors at most 1) and the diagonal 16 x 16 blocks from exact exponent differences
//         on the CUDA cores; X = T R with
//         T = (I + diag(beta) A)^-1 by forward substitution on two warps and the product on
//         tcgen05.  The scan's operands [W; Qtil], Kbar^T and Aqk go to the workspace already
//         split into bf16 hi / lo tensor-core tiles, U and e^(Gam_last) in FP32.
//   scan  (one CTA per sequence x head x 32-column block of S, the four blocks of a head one
//         cluster; chunks in order): per chunk the operand tiles arrive by bulk async copy (the
//         next chunk's while this one computes); [W; Qtil] S, then Ut = U - W S, then Kbar^T Ut
//         and Aqk Ut on tcgen05, S update in registers; the gated RMSNorm of the outputs one
//         chunk later, each token's sum of o^2 exchanged between the cluster's CTAs through
//         distributed shared memory; final state and conv window -> slot.
// Variable-length batches (cu_seqlens) take per-sequence row offsets and record indices.
// Every tensor-core product of FP32 operands sums the three bf16 products hi*hi + hi*lo + lo*hi
// (~16 significant bits per operand) in FP32 tensor memory; where the B operand is stored as one
// tile of its hi and lo halves, as two MMA passes (mma_split3_bcat / mma_split3_kcat).
#include <cstddef>

#include "kda_prefill.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

constexpr int C = kPrefillChunk;                 // 64
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kScanCols = 32;                    // columns of S per scan CTA
constexpr int kScanBlocks = kDv / kScanCols;

// Per (sequence, head, chunk) workspace record, in bytes.  Tiles are bf16 core-matrix tiles
// (see kda_tc.cuh): A1 = [W; Qtil] 128 x 128, A2 = Kbar^T 128 x 64, A3 = Aqk 64 x 64, hi then lo.
constexpr size_t kRecA1 = 0, kRecA2 = kRecA1 + 2 * 128 * 128 * 2, kRecA3 = kRecA2 + 2 * 128 * C * 2,
                 kRecU = kRecA3 + 2 * C * C * 2,          // f32 [block][t][32]
                 kRecD = kRecU + (size_t)C * 128 * 4,     // f32 [128]
                 kRecBytes = kRecD + 128 * 4;
static_assert(kRecBytes % 256 == 0, "record alignment");

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }
// Closes this thread's group of 16-byte asynchronous copies; then waits until all of its groups
// but the newest `pending` have landed.
// e^a and e^b as 2^(a log2 e) and 2^(b log2 e): one packed multiply, then the base-2
// exponential instruction (ex2.approx.f32, a few ulp) per lane.  As with the fast exponential,
// the rounding of the scaled argument adds a relative error of about |a| 2^-24.
__device__ __forceinline__ void exp_pair(float &d0, float &d1, float a, float b)
{
    constexpr float kLog2e = 1.4426950408889634f;
    float s0, s1;
    tc::mul2(s0, s1, a, b, kLog2e, kLog2e);
    asm("ex2.approx.f32 %0, %1;" : "=f"(d0) : "f"(s0));
    asm("ex2.approx.f32 %0, %1;" : "=f"(d1) : "f"(s1));
}
// x[e] *= e^(p[e] - m[e]) for 8 values, two per instruction
__device__ __forceinline__ void scale_exp_diff8(float *x, const float *p, const float *m)
{
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        float d0, d1;
        tc::sub2(d0, d1, p[e], p[e + 1], m[e], m[e + 1]);
        exp_pair(d0, d1, d0, d1);
        tc::mul2(x[e], x[e + 1], x[e], x[e + 1], d0, d1);
    }
}
template <int pending>
__device__ __forceinline__ void cp_async_commit_wait()
{
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group %0;" ::"n"(pending) : "memory");
}
__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }
// the output gate of the fused norm: fast exponential and divide (a few ulp, far below the
// BF16 rounding of the output; the norm is issue-bound with the full-precision forms)
__device__ __forceinline__ float sigmoid_fast(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

template <int W>
__device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Tokens of sequence b: its first row in the (packed) inputs and its length.  False when the
// variable-length offsets around b are inconsistent (not starting at 0, negative, decreasing,
// past the last row, or longer than the launch's bound p.T).  Whatever the offsets, a sequence
// that passes reads and writes only rows [s0, s1) of [0, total_tokens) and records below the
// workspace bound (see rec_index).
__device__ __forceinline__ bool seq_span(const RecurrentParams &p, int b, long &start, int &len)
{
    if (!p.cu_seqlens) {
        start = (long)b * p.T;
        len = p.T;
        return true;
    }
    const int s0 = __ldg(p.cu_seqlens + b), s1 = __ldg(p.cu_seqlens + b + 1);
    const int sp = b > 0 ? __ldg(p.cu_seqlens + b - 1) : 0;
    start = s0;
    len = s1 - s0;
    return s0 >= 0 && s1 >= s0 && s1 <= p.total_tokens && len <= p.T && sp <= s0 && (b > 0 || s0 == 0);
}

// Workspace record of (sequence b, head h, chunk c).  Variable lengths: chunk c of a sequence
// starting at row s is record (s / C + b + c) x H + h, which no two chunks share and which
// stays below (total / C + B) x H.
__device__ __forceinline__ size_t rec_index(const RecurrentParams &p, int b, int h, int c, int n_chunks, long start)
{
    return p.cu_seqlens ? (size_t)(start / C + b + c) * p.H + h : ((size_t)b * p.H + h) * n_chunks + c;
}

// All threads wait for an mbarrier phase; on a timeout the error is flagged and false is
// returned (the caller then frees its tensor memory and returns).
__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t parity, int *err)
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

// The same for two mbarrier phases at once, with one synchronisation.
__device__ __forceinline__ bool wait_all2(uint64_t *bar_a, uint32_t parity_a, uint64_t *bar_b, uint32_t parity_b, int *err)
{
    const bool ok = mbar_wait_bounded(bar_a, parity_a, kWaitLimitNs) && mbar_wait_bounded(bar_b, parity_b, kWaitLimitNs);
    if (__syncthreads_or(!ok)) {
        if (threadIdx.x == 0) {
            atomicOr(err, KDA_DEVERR_TIMEOUT);
            mbar_wait_bounded(bar_a, parity_a, kWaitLimitNs);
            mbar_wait_bounded(bar_b, parity_b, kWaitLimitNs);
        }
        return false;
    }
    tc::fence_after_sync();
    return true;
}

// Write one 16-byte chunk qd of a hi / lo tile pair (tile bytes `tb` apart) from 8 floats.
__device__ __forceinline__ void put_split(uint8_t *tile_hi, size_t tb, int qd, const float *x)
{
    uint4 hi, lo;
    tc::split8(x, hi, lo);
    *reinterpret_cast<uint4 *>(tile_hi + (size_t)qd * 16) = hi;
    *reinterpret_cast<uint4 *>(tile_hi + tb + (size_t)qd * 16) = lo;
}

// ============================================================================ prep

constexpr int NTA = 512;   // 16 warps: warps 0..7 own the tensor-memory phases and the solve
constexpr int kXPitch = 2 * 128 + 4;   // floats per row of the staged X = [W | U] (padded)
constexpr int kRowP = 128 + 4;         // padded row of the per-token f32 arrays: 8 consecutive
                                       // rows read 16 bytes each without bank conflicts
constexpr int kAkkP = C + 4;           // padded row of A (same reason)
constexpr int kRawRows = C + kTaps;    // pre-conv rows of one tensor: tokens t0 - 3 .. t0 + 63
constexpr size_t kRawBytes = (size_t)3 * kRawRows * kDk * 2;

// The head's conv weights (3 x 128 x 4 bf16) sit in the operand bytes past the f_b operands,
// FP8 W_fb codes (128 x 128 bytes, row-major) past those until they are converted.
constexpr int kConvWOff = 128 * 128 * 2 + C * 128 * 2;
constexpr int kW8Off = kConvWOff + 4 * 1024;

struct PrepSmem {
    // f_b operands, then Gram operands, then X = [W | U] (all in the same bytes)
    alignas(1024) uint8_t opnd[2 * 128 * 128 * 2 + 2 * 16 * 128 * 2];   // 72 KiB
    alignas(16) float q[C][kRowP];
    alignas(16) float k[C][kRowP];
    alignas(16) float v[C][kRowP];    // Aqk (same pitch) once the solve is done
    // gam, akk and raw_tail are contiguous: before the decay they hold the pre-conv bf16 rows
    // raw[tensor][row][128] (row j = token t0 - 3 + j)
    alignas(16) float gam[C][kRowP];
    alignas(16) float akk[C][kAkkP];
    alignas(16) uint8_t raw_tail[kRawBytes - sizeof(float) * C * (kRowP + kAkkP)];
    alignas(16) float beta[C];
    alignas(8) uint64_t bar;
    uint32_t tmem;
};
static_assert(C * kXPitch * 4 <= (int)sizeof(PrepSmem::opnd), "X staging fits");
static_assert(kConvWOff % 16 == 0 && kConvWOff + 3 * kDk * kConv * 2 <= (int)sizeof(PrepSmem::opnd), "conv weights fit");
static_assert(kW8Off >= kConvWOff + 3 * kDk * kConv * 2 && kW8Off % 16 == 0 &&
              kW8Off + kDk * kRank <= (int)sizeof(PrepSmem::opnd), "FP8 codes fit past the conv weights");
static_assert(offsetof(PrepSmem, akk) == offsetof(PrepSmem, gam) + sizeof(float) * C * kRowP &&
              offsetof(PrepSmem, raw_tail) == offsetof(PrepSmem, akk) + sizeof(float) * C * kAkkP &&
              sizeof(float) * C * (kRowP + kAkkP) < kRawBytes, "raw staging spans gam, akk, raw_tail");
static_assert(offsetof(PrepSmem, q) % 16 == 0 && offsetof(PrepSmem, gam) % 16 == 0 &&
              offsetof(PrepSmem, akk) % 16 == 0 && (kRowP * 4) % 16 == 0 && (kAkkP * 4) % 16 == 0 &&
              (kXPitch * 4) % 16 == 0, "float4 rows");

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }

// 8 consecutive floats as two float4 loads
__device__ __forceinline__ void ld8(const float *p, float *x)
{
    const float4 a = ld4(p), b = ld4(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// 32 columns of a product held as two halves (mma_split3_kcat): columns c .. c + 31 plus the 32
// columns `off` further, of this warp's tensor-memory lanes.
__device__ __forceinline__ void ld32_cat(uint32_t taddr, int off, float *v)
{
    float w[32];
    tc::ld32(taddr, v);
    tc::ld32(taddr + (uint32_t)off, w);
#pragma unroll
    for (int j = 0; j < 32; j += 2) tc::add2(v[j], v[j + 1], v[j], v[j + 1], w[j], w[j + 1]);
}

__global__ void __launch_bounds__(NTA, 1) kda_chunk_prep(const RecurrentParams p, uint8_t *ws, int n_chunks)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    PrepSmem &sm = *reinterpret_cast<PrepSmem *>(smem_raw);
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int H = p.H, HC = H * kDk;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    long start;
    int L;
    if (!seq_span(p, b, start, L)) {
        if (tid == 0 && c == 0 && h == 0) atomicOr(p.err_word, KDA_DEVERR_SEQLEN);
        return;
    }
    const int t0 = c * C;
    if (t0 >= L) return;   // the sequence has fewer chunks than the launch
    const int n = L - t0 < C ? L - t0 : C;
    const int slot = __ldg(p.slot_ids + b);
    if (slot < 0 || slot >= p.num_slots) {
        if (tid == 0 && c == 0 && h == 0) atomicOr(p.err_word, KDA_DEVERR_SLOT);
        return;
    }
    uint8_t *rec = ws + rec_index(p, b, h, c, n_chunks, start) * kRecBytes;
    // the token's beta logit and this thread's decay weights, read now so that their latency
    // hides behind the staging
    const float beta_logit = tid < n ? bf2f(p.beta[(size_t)(start + t0 + tid) * H + h]) : 0.f;
    const int i_row = (warp & 3) * 32 + lane, tq = warp >> 2;   // decay: channel and token block
    const float a_log = __ldg(p.A_log + h), db = __ldg(p.dt_bias + h * kDk + i_row);
    // FP8 weights: the f_b product of row i_row times the row's scale (BF16 weights: times 1)
    const float wsc = p.W_fb8 ? __ldg(p.W_fb_scale + h * kDk + i_row) : 1.0f;

    // ---- pre-conv q, k, v rows of the chunk and the 3 tokens before it (the slot's conv window
    //      before the prompt start; zeros past the prompt end), 16-byte asynchronous copies
    __nv_bfloat16 *raw = reinterpret_cast<__nv_bfloat16 *>(&sm.gam[0][0]);
    for (int qd = tid; qd < 3 * kRawRows * 16; qd += NTA) {
        const int cc = qd & 15, row = qd >> 4, tens = row / kRawRows, t = row % kRawRows - kTaps, tok = t0 + t;
        const size_t ch = (size_t)h * kDk + cc * 8;
        const __nv_bfloat16 *src = p.q + ch;   // any valid address when zero-filling
        uint32_t bytes = 0;
        if (t < n) {
            bytes = 16;
            src = tok >= 0 ? (tens == 0 ? p.q : tens == 1 ? p.k : p.v) + (size_t)(start + tok) * HC + ch
                           : p.conv_state + (((size_t)slot * 3 + tens) * kTaps + (tok + kTaps)) * HC + ch;
        }
        cp_async16(raw + (size_t)row * kDk + cc * 8, src, bytes);
    }

    // the head's conv weights [tensor][channel][tap] in operand bytes the f_b product does not
    // read; with the rows above they are the first group of copies, all that the conv waits for
    __nv_bfloat16 *cws = reinterpret_cast<__nv_bfloat16 *>(sm.opnd + kConvWOff);
    for (int qd = tid; qd < 3 * kDk * kConv / 8; qd += NTA) {   // 64 chunks of 16 bytes per tensor
        const int tens = qd >> 6, part = qd & 63;
        cp_async16(cws + (size_t)qd * 8, p.conv_w + ((size_t)tens * HC + (size_t)h * kDk) * kConv + part * 8, 16);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");

    if (warp == 0) tc::tmem_alloc(&sm.tmem, 256);
    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        fence_mbar_init();
    }
    // f_b operands, the second group: W_fb rows of the head (A, 128 x 128) and f_a of the chunk
    // (B, 64 x 128, zeros past the sequence end), waited for after the conv
    uint8_t *wcm = sm.opnd, *facm = sm.opnd + 128 * 128 * 2;
    const bool fp8 = p.W_fb8 != nullptr;   // FP8 E4M3 codes with per-row scales
    if (!fp8) {
        for (int qd = tid; qd < 128 * 16; qd += NTA) {
            int r, k;
            tc::cm_chunk(qd, 128, r, k);
            cp_async16(wcm + qd * 16, p.W_fb + ((size_t)h * kDk + r) * kRank + k, 16);
        }
    } else {
        // the codes land row-major in free operand bytes and become bf16 tiles (exactly) below
        for (int qd = tid; qd < 128 * 128 / 16; qd += NTA)
            cp_async16(sm.opnd + kW8Off + qd * 16, p.W_fb8 + (size_t)h * kDk * kRank + qd * 16, 16);
    }
    for (int qd = tid; qd < C * 16; qd += NTA) {
        int r, k;
        tc::cm_chunk(qd, 128, r, k);
        cp_async16(facm + qd * 16, r < n ? p.f_a + (size_t)(start + t0 + r) * kRank + k : p.f_a, r < n ? 16 : 0);
    }
    cp_async_commit_wait<1>();   // this thread's rows and conv weights
    __syncthreads();

    // ---- short causal conv + SiLU from the staged rows: an item is 2 channels x 8 tokens of
    //      one tensor (a warp covers 64 channels of one run), three items per thread
    for (int it = tid; it < 3 * (C / 8) * 64; it += NTA) {
        const int c2 = (it & 63) * 2, rest = it >> 6, tens = rest % 3, tr = rest / 3;
        const uint4 wv = *reinterpret_cast<const uint4 *>(cws + ((size_t)tens * kDk + c2) * kConv);
        const uint32_t wu[4] = {wv.x, wv.y, wv.z, wv.w};
        float w[2][kConv];   // [channel][tap]
#pragma unroll
        for (int e = 0; e < 2; e++) {
            w[e][0] = __uint_as_float(wu[2 * e] << 16);
            w[e][1] = __uint_as_float(wu[2 * e] & 0xffff0000u);
            w[e][2] = __uint_as_float(wu[2 * e + 1] << 16);
            w[e][3] = __uint_as_float(wu[2 * e + 1] & 0xffff0000u);
        }
        float x[11][2];
        const __nv_bfloat16 *rp = raw + ((size_t)tens * kRawRows + tr * 8) * kDk + c2;
#pragma unroll
        for (int j = 0; j < 11; j++) {
            const uint32_t u = *reinterpret_cast<const uint32_t *>(rp + (size_t)j * kDk);
            x[j][0] = __uint_as_float(u << 16);
            x[j][1] = __uint_as_float(u & 0xffff0000u);
        }
        float *dst = tens == 0 ? &sm.q[0][0] : tens == 1 ? &sm.k[0][0] : &sm.v[0][0];
#pragma unroll
        for (int e = 0; e < 8; e++) {
            const int t = tr * 8 + e;
            // both channels at once, tap by tap (the same rounding as one fmaf chain each)
            float o[2];
            tc::mul2(o[0], o[1], w[0][0], w[1][0], x[e][0], x[e][1]);
#pragma unroll
            for (int j = 1; j < kConv; j++)
                tc::fma2(o[0], o[1], w[0][j], w[1][j], x[e + j][0], x[e + j][1], o[0], o[1]);
#pragma unroll
            for (int ch = 0; ch < 2; ch++) o[ch] = t < n ? __fdividef(o[ch], 1.0f + __expf(-o[ch])) : 0.f;
            *reinterpret_cast<float2 *>(dst + t * kRowP + c2) = make_float2(o[0], o[1]);
        }
    }
    if (tid < C) sm.beta[tid] = tid < n ? sigmoidf_(beta_logit) : 0.f;
    cp_async_commit_wait<0>();   // this thread's f_b operand copies
    if (fp8) {
        __syncthreads();   // every thread's codes have landed
        for (int qd = tid; qd < 128 * 16; qd += NTA) {
            int r, k;
            tc::cm_chunk(qd, 128, r, k);
            float w[8];
            e4m3x8_to_f32(*reinterpret_cast<const uint2 *>(sm.opnd + kW8Off + r * kRank + k), w);
            *reinterpret_cast<uint4 *>(wcm + qd * 16) =
                make_uint4(tc::pack2(__float2bfloat16_rn(w[0]), __float2bfloat16_rn(w[1])),
                           tc::pack2(__float2bfloat16_rn(w[2]), __float2bfloat16_rn(w[3])),
                           tc::pack2(__float2bfloat16_rn(w[4]), __float2bfloat16_rn(w[5])),
                           tc::pack2(__float2bfloat16_rn(w[6]), __float2bfloat16_rn(w[7])));
        }
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
    // ---- q, k L2 norms (q also scaled by dk^-1/2); rows 0..63 q, 64..127 k
    for (int row = warp; row < 2 * C; row += NTA / 32) {
        float *x = row < C ? &sm.q[row][0] : &sm.k[row - C][0];
        float4 a = ld4(x + lane * 4);
        float s0, s1;
        tc::mul2(s0, s1, a.x, a.y, a.x, a.y);
        tc::fma2(s0, s1, a.z, a.w, a.z, a.w, s0, s1);
        const float ss = group_sum<32>(s0 + s1);
        const float f = (row < C ? rsqrtf((float)kDk) : 1.0f) * rsqrtf(ss + p.l2_eps);
        tc::mul2(a.x, a.y, a.x, a.y, f, f);
        tc::mul2(a.z, a.w, a.z, a.w, f, f);
        st4(x + lane * 4, a);
    }
    // ---- decay: TMEM holds graw[i = lane row][t = column]; warp w takes channels of lane
    //      quarter w % 4 for the 16 tokens of block w / 4, then adds the totals of the blocks
    //      before it (scratch over the A bytes, not yet in use)
    bool ok = wait_all(&sm.bar, phase, p.err_word);
    phase ^= 1;
    float *totals = &sm.akk[0][0];   // [4][128]
    if (ok) {
        float g[16];
        tc::ld16(tc::taddr(tmem, (warp & 3) * 32, 16 * tq), g);
        const float a = expf(a_log);
        float G = 0.f;
        bool finite = true;
#pragma unroll
        for (int tt = 0; tt < 16; tt += 2) {
            // -a softplus(graw wsc + dt_bias) for two tokens, the arithmetic around the
            // exponential and logarithm packed (2^(x log2 e) and the fast logarithm: absolute
            // error about 1e-7 in the log-decay, a relative error of that size in each decay
            // factor; the token-serial kernels keep the full-precision form)
            float x0, x1, e0, e1, g0, g1;
            tc::fma2(x0, x1, g[tt], g[tt + 1], wsc, wsc, db, db);
            exp_pair(e0, e1, x0, x1);
            tc::add2(e0, e1, e0, e1, 1.0f, 1.0f);
            g0 = x0 > 20.0f ? x0 : __logf(e0);
            g1 = x1 > 20.0f ? x1 : __logf(e1);
            tc::mul2(g0, g1, g0, g1, -a, -a);
            const int t = 16 * tq + tt;
            if (t >= n) g0 = 0.f;
            if (t + 1 >= n) g1 = 0.f;
            finite &= isfinite(g0) && isfinite(g1);
            G += g0;
            sm.gam[t][i_row] = G;
            G += g1;
            sm.gam[t + 1][i_row] = G;
        }
        if (!finite) atomicOr(p.err_word, KDA_DEVERR_DECAY);
        totals[tq * 128 + i_row] = G;
    }
    __syncthreads();
    if (ok && tq > 0) {
        float off = totals[i_row];
        for (int j = 1; j < tq; j++) off += totals[j * 128 + i_row];
#pragma unroll
        for (int tt = 0; tt < 16; tt++) sm.gam[16 * tq + tt][i_row] += off;
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---- gated Gram blocks: A operand rows [k; q] (128 x 128 channels) scaled by e^(Gam_t - Gam_ref),
    //      B operand keys scaled by e^(Gam_ref - Gam_s); the two factors multiply to the exact
    //      gating e^(Gam_t - Gam_s) of every kept entry.  Entries with t < s (or t <= s for A)
    //      may overflow; the A and Aqk reads below discard them with a select.
    uint8_t *ahi = sm.opnd, *bhi = sm.opnd + 2 * 128 * 128 * 2;
    const size_t atb = 128 * 128 * 2, btb = 16 * 128 * 2;
    // One reference (token 31) serves the whole chunk when every channel's log-decay stays
    // within 64 of it (factors within e^(+-64), far from FP32 / BF16 overflow and subnormals):
    // A is staged once and two N = 32 products (B over the bytes of A, not yet in use) fill
    // all 64 columns.  Otherwise (the wide form below) no factor exceeds 1.
    const bool wide = __syncthreads_or(tid < 128 && (sm.gam[0][tid] - sm.gam[31][tid] > 64.f ||
                                                     sm.gam[31][tid] - sm.gam[C - 1][tid] > 64.f));
    if (ok && !wide) {
        const int kg = (tid >> 3) & 15, k = kg * 8;
        float gr[8];
        ld8(&sm.gam[31][k], gr);
        for (int idx = tid; idx < 2 * C * 16; idx += NTA) {
            const int rl = (idx >> 7) * 8 + (idx & 7), half = rl >= C, t = half ? rl - C : rl;
            const int qd = (rl >> 3) * 128 + kg * 8 + (rl & 7);
            float x[8], gt[8];
            ld8(half ? &sm.q[t][k] : &sm.k[t][k], x);
            ld8(&sm.gam[t][k], gt);
            scale_exp_diff8(x, gt, gr);
            put_split(ahi, atb, qd, x);
        }
        uint8_t *b32 = reinterpret_cast<uint8_t *>(&sm.akk[0][0]);   // keys of 32 tokens, hi / lo
        constexpr size_t b32b = (size_t)32 * 128 * 2;
        static_assert(2 * b32b <= sizeof(PrepSmem::akk), "B operand fits");
        // (the second B reuses the bytes of the first: the wait on the first product's commit
        // orders that reuse)
        for (int half32 = 0; half32 < 2 && ok; half32++) {
            {
                // 512 chunks, a warp taking 32 consecutive tokens of one 8-channel group
                const int r = tid & 31, kb = warp * 8, s = 32 * half32 + r;
                float x[8], gs[8], grb[8];
                ld8(&sm.k[s][kb], x);
                ld8(&sm.gam[s][kb], gs);
                ld8(&sm.gam[31][kb], grb);
                scale_exp_diff8(x, grb, gs);
                put_split(b32, b32b, (r >> 3) * 128 + (kb >> 3) * 8 + (r & 7), x);
            }
            tc::fence_smem_to_async();
            tc::fence_before_sync();
            __syncthreads();
            tc::fence_after_sync();
            if (tid == 0) {
                tc::mma_split3_kcat(tmem + 64 + 64 * half32, smem_u32(ahi), smem_u32(ahi + atb), 128, smem_u32(b32),
                                    128, 32, 8, false);
                tc::commit(&sm.bar);
            }
            ok = wait_all(&sm.bar, phase, p.err_word);
            phase ^= 1;
        }
    }
    // Wide decay range: the blocks below the diagonal (tokens t of a later 16-token block than
    // the keys s) are referenced to the last token b of the key block, so that both factors,
    // e^(Gam_t - Gam_b) and e^(Gam_b - Gam_s), lie in (0, 1] whatever the decay: one N = 16
    // product per key block, over the rows t > b.  The rows of earlier blocks keep whatever an
    // earlier round left (finite factors at most 1, or bytes of an earlier phase); their
    // products fall on entries that the read-outs below discard or replace.
    for (int J = 0; J < 3 && ok && wide; J++) {
        const int bref = 16 * J + 15, t_lo = 16 * (J + 1), span = C - t_lo;
        const int kg = (tid >> 3) & 15, k = kg * 8;   // the same 8 channels in every iteration
        static_assert(NTA % 128 == 0, "fixed channel group per thread");
        float gb[8];
        ld8(&sm.gam[bref][k], gb);
        for (int idx = tid; idx < 2 * span * 16; idx += NTA) {
            const int rl = (idx >> 7) * 8 + (idx & 7);
            const int half = rl >= span, t = t_lo + (half ? rl - span : rl), r = half * C + t;
            const int qd = (r >> 3) * 128 + kg * 8 + (r & 7);
            float x[8], gt[8];
            ld8(half ? &sm.q[t][k] : &sm.k[t][k], x);
            ld8(&sm.gam[t][k], gt);
#pragma unroll
            for (int e = 0; e < 8; e++) x[e] *= __expf(gt[e] - gb[e]);
            put_split(ahi, atb, qd, x);
        }
        for (int qd = tid; qd < 16 * 16; qd += NTA) {
            int r, kb;
            tc::cm_chunk(qd, 128, r, kb);
            const int j = 16 * J + r;
            float x[8], gj[8], gbb[8];
            ld8(&sm.k[j][kb], x);
            ld8(&sm.gam[j][kb], gj);
            ld8(&sm.gam[bref][kb], gbb);
#pragma unroll
            for (int e = 0; e < 8; e++) x[e] *= __expf(gbb[e] - gj[e]);
            put_split(bhi, btb, qd, x);
        }
        tc::fence_smem_to_async();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (tid == 0) {
            tc::mma_split3(tmem + 64 + 16 * J, smem_u32(ahi), smem_u32(ahi + atb), 128, smem_u32(bhi),
                           smem_u32(bhi + btb), 128, 16, 8, false);
            tc::commit(&sm.bar);
        }
        ok = wait_all(&sm.bar, phase, p.err_word);
        phase ^= 1;
    }
    // Wide decay range, the diagonal 16-token blocks: A[t][s] (s < t) and Aqk[t][s] (s <= t)
    // from the exact exponent differences e^(Gam_t - Gam_s) <= 1 on the CUDA cores, into the
    // B operand bytes (free now): dA [block][t][s], then dQ [block][t][s].  An item is one
    // (block, t, s) with s <= t; 8 lanes share it, lane l taking channels 4 l + 32 i.
    float *diag = reinterpret_cast<float *>(bhi);
    static_assert(2 * 4 * 16 * 16 * 4 <= 2 * btb, "diagonal blocks fit the B operand bytes");
    if (ok && wide) {
        const int sub = lane & 7;
        for (int it = warp * 4 + (lane >> 3); it < 4 * 136; it += NTA / 8) {
            const int J = it / 136;
            int rem = it % 136, tl = 0;
            while (rem > tl) { rem -= tl + 1; tl++; }   // (tl, sl = rem), sl <= tl < 16
            const int t = 16 * J + tl, s_ = 16 * J + rem;
            float a_kk = 0.f, a_qk = 0.f;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int c = 4 * sub + 32 * i;
                const float4 gt = ld4(&sm.gam[t][c]), gs = ld4(&sm.gam[s_][c]);
                const float4 kt = ld4(&sm.k[t][c]), ks = ld4(&sm.k[s_][c]), qt = ld4(&sm.q[t][c]);
                const float e0 = __expf(gt.x - gs.x) * ks.x, e1 = __expf(gt.y - gs.y) * ks.y;
                const float e2 = __expf(gt.z - gs.z) * ks.z, e3 = __expf(gt.w - gs.w) * ks.w;
                a_kk = fmaf(kt.x, e0, fmaf(kt.y, e1, fmaf(kt.z, e2, fmaf(kt.w, e3, a_kk))));
                a_qk = fmaf(qt.x, e0, fmaf(qt.y, e1, fmaf(qt.z, e2, fmaf(qt.w, e3, a_qk))));
            }
            a_kk = group_sum<8>(a_kk);
            a_qk = group_sum<8>(a_qk);
            if (sub == 0) {
                diag[(J * 16 + tl) * 16 + rem] = rem < tl ? a_kk : 0.f;
                diag[1024 + (J * 16 + tl) * 16 + rem] = a_qk;
            }
        }
    }
    static_assert((4 * 136) % 4 == 0, "every lane group of a warp takes the same number of items");
    if (wide) {
        // the diagonal blocks are written (the one-reference form ended in the products' wait)
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
    }
    // lanes 0..63 of columns 64.. hold A[i][j] (kept for j < i)
    const int wq = warp & 3, half = warp >> 2;
    if (ok && warp < 8 && wq < 2) {
        float g[32];
        if (wide) tc::ld32(tc::taddr(tmem, 32 * wq, 64 + 32 * half), g);
        else ld32_cat(tc::taddr(tmem, 32 * wq, 64 + 64 * half), 32, g);
        const int row = 32 * wq + lane;
#pragma unroll
        for (int j4 = 0; j4 < 32; j4 += 4) {
            const int j = 32 * half + j4;
            float x[4];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                x[e] = j + e < row ? g[j4 + e] : 0.f;
                if (wide && j + e < row && ((j + e) >> 4) == (row >> 4))
                    x[e] = diag[((row >> 4) * 16 + (row & 15)) * 16 + ((j + e) & 15)];
            }
            st4(&sm.akk[row][j], make_float4(x[0], x[1], x[2], x[3]));
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---- X = [W | U] = T R with T = (I + diag(beta) A)^-1 and R = diag(beta) [Ktil | V]:
    //      warps 0, 1 compute T one column per thread by forward substitution (four interleaved
    //      partial sums per dot product); warps 2..7 meanwhile stage R^T [256 x 64] as a bf16
    //      hi / lo operand over the operand bytes; warps 8..15 write the operand tiles that do
    //      not depend on X: the Qtil rows of A1, A2 = Kbar^T, e^(Gam_last), and (warps 10, 11,
    //      which see tensor-memory lanes 64..127) A3 = Aqk straight from tensor memory.
    //      Then T goes through an FP32 transpose (over the bytes of A) into a bf16 hi / lo
    //      operand (over those of v) and two tensor-core products give X^T in tensor memory
    //      columns 128..255, from where X lands in the staging rows xs (over R^T).
    float *xs = reinterpret_cast<float *>(sm.opnd);
    uint8_t *rt = sm.opnd;                           // R^T hi [256 x 64], then lo
    constexpr size_t rtb = (size_t)256 * C * 2;
    float *tT = &sm.akk[0][0];                       // T, FP32, [t][65]
    constexpr int kTP = C + 1;
    uint8_t *tops = reinterpret_cast<uint8_t *>(&sm.v[0][0]);   // T hi [64 x 64], then lo
    constexpr size_t tob = (size_t)C * C * 2;
    static_assert(2 * rtb <= sizeof(PrepSmem::opnd) && (size_t)C * kTP * 4 <= sizeof(PrepSmem::akk) &&
                  2 * tob <= sizeof(PrepSmem::v), "solve operands fit");
    uint8_t *a1 = rec + kRecA1, *a2 = rec + kRecA2, *a3 = rec + kRecA3;
    float *urec = reinterpret_cast<float *>(rec + kRecU), *drec = reinterpret_cast<float *>(rec + kRecD);
    float y[C];                                      // warps 0, 1: column tid of T
    if (ok && warp < 2) {
        const int j = tid;
#pragma unroll
        for (int t = 0; t < C; t++) {
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int s4 = 0; s4 < t / 4; s4++) {
                const float4 A = ld4(&sm.akk[t][4 * s4]);   // four sums, two per instruction
                tc::fma2(a0, a1, A.x, A.y, y[4 * s4], y[4 * s4 + 1], a0, a1);
                tc::fma2(a2, a3, A.z, A.w, y[4 * s4 + 2], y[4 * s4 + 3], a2, a3);
            }
#pragma unroll
            for (int s = (t / 4) * 4; s < t; s++) a0 = fmaf(sm.akk[t][s], y[s], a0);
            y[t] = (t == j ? 1.f : 0.f) - sm.beta[t] * ((a0 + a1) + (a2 + a3));
        }
        // T in FP32 over the bytes of A, which only these two warps read in this phase
        named_bar_sync(1, 2 * 32);
#pragma unroll
        for (int t = 0; t < C; t++) tT[t * kTP + tid] = y[t];
    } else if (ok && warp < 8) {
        // R^T: element (column c, token s) = beta_s Ktil_s[c] (c < 128) or beta_s v_s[c - 128];
        // a warp covers 32 consecutive columns of one 8-token group
        for (int idx = tid - 64; idx < 256 * (C / 8); idx += 192) {
            const int col = idx & 255, sg = idx >> 8, s0 = sg * 8;
            float x[8];
            if (col < 128) {
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    float f0, f1;
                    tc::mul2(x[e], x[e + 1], sm.beta[s0 + e], sm.beta[s0 + e + 1], sm.k[s0 + e][col], sm.k[s0 + e + 1][col]);
                    exp_pair(f0, f1, sm.gam[s0 + e][col], sm.gam[s0 + e + 1][col]);
                    tc::mul2(x[e], x[e + 1], x[e], x[e + 1], f0, f1);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; e++) x[e] = sm.beta[s0 + e] * sm.v[s0 + e][col - 128];
            }
            put_split(rt, rtb, (col >> 3) * C + sg * 8 + (col & 7), x);
        }
    } else if (ok) {
        const int wt = tid - 256;   // 0..255
        // A1 rows 64..127: Qtil = q e^(Gam)
        for (int qd = 1024 + wt; qd < 128 * 16; qd += 256) {
            int r, k;
            tc::cm_chunk(qd, 128, r, k);
            const int t = r - C;
            float x[8], g[8];
            ld8(&sm.q[t][k], x);
            ld8(&sm.gam[t][k], g);
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                float f0, f1;
                exp_pair(f0, f1, g[e], g[e + 1]);
                tc::mul2(x[e], x[e + 1], x[e], x[e + 1], f0, f1);
            }
            put_split(a1, 128 * 128 * 2, qd, x);
        }
        // A2 = Kbar^T (128 x 64): element (i, t) = k_t[i] e^(Gam_last[i] - Gam_t[i]); a warp
        // takes 32 consecutive channels i of one 8-token group
        for (int idx = wt; idx < 128 * (C / 8); idx += 256) {
            const int i = idx & 127, tg = idx >> 7, t = tg * 8;
            const int qd = (i >> 3) * C + tg * 8 + (i & 7);
            const float gl = sm.gam[C - 1][i];   // padded tokens keep Gam constant
            float x[8], g[8], gls[8];
#pragma unroll
            for (int e = 0; e < 8; e++) {
                x[e] = sm.k[t + e][i];
                g[e] = sm.gam[t + e][i];
                gls[e] = gl;
            }
            scale_exp_diff8(x, gls, g);
            put_split(a2, 128 * C * 2, qd, x);
        }
        if (wt < 128) drec[wt] = __expf(sm.gam[C - 1][wt]);
        // A3 = Aqk (64 x 64): tensor-memory lane 64 + t, column 64 + j holds Aqk[t][j] (j <= t kept)
        if (warp == 10 || warp == 11) {
            const int t = 32 * (warp - 10) + lane;
#pragma unroll
            for (int hf = 0; hf < 2; hf++) {
                float g[32];
                if (wide) tc::ld32(tc::taddr(tmem, 32 * (warp & 3), 64 + 32 * hf), g);
                else ld32_cat(tc::taddr(tmem, 32 * (warp & 3), 64 + 64 * hf), 32, g);
#pragma unroll
                for (int j8 = 0; j8 < 4; j8++) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        const int j = 32 * hf + 8 * j8 + e;
                        x[e] = j <= t ? g[8 * j8 + e] : 0.f;
                        if (wide && j <= t && (j >> 4) == (t >> 4)) x[e] = diag[1024 + ((t >> 4) * 16 + (t & 15)) * 16 + (j & 15)];
                    }
                    put_split(a3, C * C * 2, (t >> 3) * C + (4 * hf + j8) * 8 + (t & 7), x);
                }
            }
        }
    }
    __syncthreads();   // T is complete; k, v and gam readers of the phase are done
    // T as the B operand (N = 64 tokens t, K = 64 tokens s): one 16-byte chunk per thread
    if (ok) {
        const int t = tid & (C - 1), sg = tid >> 6;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; e++) x[e] = tT[t * kTP + sg * 8 + e];
        put_split(tops, tob, (t >> 3) * C + sg * 8 + (t & 7), x);
    }
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (ok && tid == 0) {
        // X^T[c][t] = sum_s R^T[c][s] T[t][s]: columns c = 0..127 -> tmem 0.., 128..255 -> 128..,
        // each product as two halves of 64 columns (see mma_split3_kcat); the f_b and Gram
        // results these columns held have been read
        tc::mma_split3_kcat(tmem, smem_u32(rt), smem_u32(rt + rtb), C, smem_u32(tops), C, C, C / 16, false);
        tc::mma_split3_kcat(tmem + 128, smem_u32(rt) + 128 * C * 2, smem_u32(rt + rtb) + 128 * C * 2, C,
                            smem_u32(tops), C, C, C / 16, false);
        tc::commit(&sm.bar);
    }
    if (ok) {
        ok = wait_all(&sm.bar, phase, p.err_word);
        phase ^= 1;
    }
    // X from tensor memory into the staging rows: warp w reads lane quarter w % 4 of product
    // (w / 4) % 2, tokens 32 (w / 8) ..
    if (ok) {
        const int q4 = warp & 3, prod = (warp >> 2) & 1, th = warp >> 3;
        float g[32];
        ld32_cat(tc::taddr(tmem, 32 * q4, 128 * prod + 32 * th), 64, g);
        const int col = 128 * prod + 32 * q4 + lane;
#pragma unroll
        for (int tt = 0; tt < 32; tt++) xs[(32 * th + tt) * kXPitch + col] = g[tt];
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();   // the deallocation follows every warp's tensor-memory loads
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
    if (!ok) return;

    // ---- X-dependent operands: A1 rows 0..63 = W, and U column-block major [block][t][32]
    for (int qd = tid; qd < 1024; qd += NTA) {
        int r, k;
        tc::cm_chunk(qd, 128, r, k);
        float x[8];
        ld8(xs + r * kXPitch + k, x);
        put_split(a1, 128 * 128 * 2, qd, x);
    }
    // U, column-block major: [block][t][32], the 16-byte chunks of row t rotated by t % 8 (chunk
    // g of the row at position g ^ (t % 8)), so that the scan's threads, one per token, read
    // their own rows without bank conflicts
    for (int idx = tid; idx < C * 128 / 4; idx += NTA) {
        const int t = idx / 32, c4 = (idx % 32) * 4, blk = c4 / kScanCols, cc = c4 % kScanCols;
        st4(urec + ((size_t)blk * C + t) * kScanCols + (((cc >> 2) ^ (t & 7)) << 2), ld4(xs + t * kXPitch + 128 + c4));
    }
}

// ============================================================================ scan

constexpr int NTB = 256;
constexpr int kHalfCols = kScanCols / 2;   // columns of S per thread
constexpr int kScanTmemCols = 256;         // two [W S; O] accumulators and Kbar^T Ut, 64 columns each
constexpr int kNormDepth = 4;              // chunks of per-token sums of o^2 in flight between a head's CTAs

// One chunk's K = tokens operands, double-buffered so that the next chunk's copies are issued
// while this chunk's first product runs.  The [.; Aqk] operand of the second product is 128 rows:
// rows 64..127 are Aqk, rows 0..63 whatever precedes it in this struct (the hi tile starts 8 KiB
// before aqk[0], inside a2's lo tile; the lo tile starts at aqk[0]).  Those rows only add to
// rows 0..63 of the product's accumulator, W S, which has been read before the product is issued
// and is not read again; every byte they read is finite data of the same chunk.
struct ScanRest {
    alignas(1024) uint8_t a2[2][128 * C * 2];           // Kbar^T hi / lo, K = tokens
    uint8_t aqk[2][C * C * 2];                          // Aqk hi / lo (rows 64..127 of [.; Aqk])
    alignas(16) float u[C][kScanCols];                  // U, this CTA's columns (chunks rotated by t % 8)
    alignas(16) float d[128];                           // e^(Gam_last)
};
static_assert(offsetof(ScanRest, aqk) == 2 * 128 * C * 2 && C * C * 2 <= 128 * C * 2,
              "the rows before each Aqk tile lie inside the struct");
struct ScanSmem {
    alignas(1024) uint8_t a1[2][128 * 128 * 2];         // [W; Qtil] hi / lo, K = dk
    ScanRest rest[2];
    alignas(1024) uint8_t b1[2 * kScanCols * 128 * 2];  // [S^T hi | S^T lo], N = 64, K = dk, MN-major
    alignas(1024) uint8_t b2[2 * kScanCols * C * 2];    // [Ut^T hi | Ut^T lo], N = 64, K = tokens, MN-major
    // per token, each column block's sum of o^2 over its 32 columns, written by every CTA of the
    // cluster into every other (chunk c in buffer c % kNormDepth), and this CTA's second column
    // half's sums handed to the first half's threads
    alignas(16) float part[kNormDepth][kScanBlocks][C];
    alignas(16) float half_ss[C];
    alignas(8) uint64_t bar_mma, bar_a1, bar_rest[2], bar_part[kNormDepth];
    uint32_t tmem;
};
static_assert(sizeof(ScanSmem) <= 227 * 1024, "scan shared memory");

// 8 columns c0 .. c0 + 7 of k-row k of a [B hi | B lo] operand (MN-major, N = 2 x 32), from 8
// floats: the hi chunk among the first 32 columns, the lo chunk 32 columns further.
__device__ __forceinline__ void put_cat(uint8_t *b, int c0, int k, const float *x)
{
    uint4 hi, lo;
    tc::split8(x, hi, lo);
    *reinterpret_cast<uint4 *>(b + tc::bmn_off(c0, k, 2 * kScanCols)) = hi;
    *reinterpret_cast<uint4 *>(b + tc::bmn_off(kScanCols + c0, k, 2 * kScanCols)) = lo;
}

// 16 columns of a product held as two halves (mma_split3_bcat): columns c .. c + 15 plus
// columns 32 + c .. 32 + c + 15 of this warp's tensor-memory lanes.
__device__ __forceinline__ void ld_cat(uint32_t taddr, float *v)
{
    float w[kHalfCols];
    tc::ld16(taddr, v);
    tc::ld16(taddr + kScanCols, w);
#pragma unroll
    for (int j = 0; j < kHalfCols; j += 2) tc::add2(v[j], v[j + 1], v[j], v[j + 1], w[j], w[j + 1]);
}

template <typename ST>
__global__ void __launch_bounds__(NTB, 1) kda_chunk_scan(const RecurrentParams p, const uint8_t *ws, int n_chunks)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    ScanSmem &sm = *reinterpret_cast<ScanSmem *>(smem_raw);
    const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int H = p.H, HC = H * kDk;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // warp w sees tensor-memory lanes 32 (w % 4) ..; it owns row (or token) 32 (w % 4) + lane and
    // the half w / 4 of the CTA's 32 columns
    const int quarter = warp & 3, row = 32 * quarter + lane, cofs = kHalfCols * (warp >> 2);
    long start;
    int L;
    if (!seq_span(p, b, start, L)) return;         // flagged by the prep launch
    if (L == 0) return;                            // nothing to add: state and window stay
    const int slot = __ldg(p.slot_ids + b);
    if (slot < 0 || slot >= p.num_slots) return;   // flagged by the prep launch
    const int col0 = blk * kScanCols;
    const int nc = (L + C - 1) / C;                // this sequence's chunks

    // one thread starts the copies of chunk c's tiles
    // (hi and lo lie back to back in the record and in shared memory: one copy)
    auto issue_a1 = [&](int c) {
        const uint8_t *rec = ws + rec_index(p, b, h, c, n_chunks, start) * kRecBytes;
        mbar_arrive_expect_tx(&sm.bar_a1, 2 * 128 * 128 * 2);
        bulk_load(sm.a1[0], rec + kRecA1, 2 * 128 * 128 * 2, &sm.bar_a1);
    };
    // (the record keeps Kbar^T hi and lo, and Aqk hi and lo, back to back: one copy each)
    auto issue_rest = [&](int c, int bf) {
        const uint8_t *rec = ws + rec_index(p, b, h, c, n_chunks, start) * kRecBytes;
        ScanRest &r = sm.rest[bf];
        mbar_arrive_expect_tx(&sm.bar_rest[bf], 2 * 128 * C * 2 + 2 * C * C * 2 + C * kScanCols * 4 + 128 * 4);
        bulk_load(r.a2[0], rec + kRecA2, 2 * 128 * C * 2, &sm.bar_rest[bf]);
        bulk_load(r.aqk[0], rec + kRecA3, 2 * C * C * 2, &sm.bar_rest[bf]);
        bulk_load(&r.u[0][0], rec + kRecU + (size_t)blk * C * kScanCols * 4, C * kScanCols * 4, &sm.bar_rest[bf]);
        bulk_load(r.d, rec + kRecD, 128 * 4, &sm.bar_rest[bf]);
    };

    if (warp == 0) tc::tmem_alloc(&sm.tmem, kScanTmemCols);
    if (tid == 0) {
        mbar_init(&sm.bar_mma, 1);
        mbar_init(&sm.bar_a1, 1);
        mbar_init(&sm.bar_rest[0], 1);
        mbar_init(&sm.bar_rest[1], 1);
        for (int q = 0; q < kNormDepth; q++) mbar_init(&sm.bar_part[q], 1);
        fence_mbar_init();
        // each use of a sums buffer: this arrival plus the 4-byte sums of the cluster's CTAs
        for (int q = 0; q < kNormDepth; q++) mbar_arrive_expect_tx(&sm.bar_part[q], kScanBlocks * C * 4);
        issue_a1(0);
        issue_rest(0, 0);
    }
    // every CTA of the cluster has initialised its barriers before another arrives on them
    cluster_arrive();
    // S row `row`, columns col0 + cofs .. + 15, FP32 in registers
    ST *tile = reinterpret_cast<ST *>(p.state) + ((size_t)slot * H + h) * (kDk * kDv);
    float S[kHalfCols];
#pragma unroll
    for (int j = 0; j < kHalfCols; j++) S[j] = (float)tile[(size_t)row * kDv + col0 + cofs + j];
    // row i of S is k-row i of the B operand [S^T hi | S^T lo] (MN-major, N = 64: the bf16 hi
    // parts of the 32 columns, then their lo parts), as 16-byte chunks, each written by the
    // thread that holds those 8 columns of the row
    auto put_state = [&]() {
#pragma unroll
        for (int g = 0; g < kHalfCols / 8; g++)
            put_cat(sm.b1, cofs + 8 * g, row, &S[8 * g]);
    };
    // The gated RMSNorm of the outputs, on the warps of lane quarters 2 and 3 (token
    // t = 32 (quarter - 2) + lane of a chunk, this thread's 16 columns), which read a chunk's
    // outputs from [. ; O] (tensor-memory lanes 64..127) while the next chunk's first product
    // runs.  The four CTAs of the cluster hold the four 32-column blocks of the head: each sends
    // every token's sum of o^2 over its block into part[chunk % kNormDepth][its rank] of all four
    // (asynchronous stores that count their bytes on the receivers' bar_part of that buffer), and
    // finishes a chunk one chunk later, once all four sums are in.  A chunk's sums are read before
    // the next chunk's are sent, so a buffer is written again only after every CTA has read it.
    float nw[kHalfCols];
    if (quarter >= 2) {
#pragma unroll
        for (int j = 0; j < kHalfCols; j++) nw[j] = __ldg(p.norm_w + col0 + cofs + j);
    }
    auto norm_send = [&](int cc, const float *o) {
        const int t = row - C, q = cc % kNormDepth;
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < kHalfCols; j++) ss = fmaf(o[j], o[j], ss);
        if (cofs != 0) sm.half_ss[t] = ss;
        named_bar_sync(1, 4 * 32);   // the four warps of lane quarters 2 and 3
        if (cofs == 0) {
            ss += sm.half_ss[t];
#pragma unroll
            for (int r = 0; r < kScanBlocks; r++)
                st_async_f32(map_to_rank(&sm.part[q][blk][t], (uint32_t)r), ss, map_to_rank(&sm.bar_part[q], (uint32_t)r));
        }
    };
    auto load_gate = [&](int cc, uint4 *g) {
        const int t = row - C, t0 = cc * C, n = L - t0 < C ? L - t0 : C;
        if (t < n) {
            const uint4 *src = reinterpret_cast<const uint4 *>(p.gate + (size_t)(start + t0 + t) * HC + h * kDv + col0 + cofs);
            g[0] = __ldg(src);
            g[1] = __ldg(src + 1);
        }
    };
    // chunk cc's four sums for this thread's token -> 1 / rms, or a negative value when they did
    // not arrive in time (flagged; the thread then waits for no later chunk's sums either, so a
    // failed CTA costs its peers one bounded wait, not one per chunk); the first thread re-arms
    // the buffer for its next use
    bool norm_live = true;
    auto norm_read = [&](int cc) {
        const int t = row - C, q = cc % kNormDepth;
        if (!norm_live) return -1.0f;
        if (!mbar_wait_bounded<true>(&sm.bar_part[q], (uint32_t)(cc / kNormDepth) & 1u, kWaitLimitNs)) {
            atomicOr(p.err_word, KDA_DEVERR_TIMEOUT);
            norm_live = false;
            return -1.0f;
        }
        const float ms = ((sm.part[q][0][t] + sm.part[q][1][t]) + (sm.part[q][2][t] + sm.part[q][3][t])) * (1.0f / kDv);
        if (tid == 2 * 32) mbar_arrive_expect_tx(&sm.bar_part[q], kScanBlocks * C * 4);
        return rsqrtf(ms + p.norm_eps);
    };
    // the outputs of 8 of this thread's 16 columns (part 0: the first 8, part 1: the others)
    auto norm_finish = [&](int cc, const float *o, const uint4 *g, float rr, int part) {
        const int t = row - C, t0 = cc * C, n = L - t0 < C ? L - t0 : C;
        if (t >= n || rr < 0.f) return;
        const uint4 gp = g[part];
        const uint32_t gw[4] = {gp.x, gp.y, gp.z, gp.w};
        uint32_t yw[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const int j = 8 * part + 2 * e;
            // ((o rr) w_norm) sigmoid(gate), two columns per instruction
            float y0, y1;
            tc::mul2(y0, y1, o[j], o[j + 1], rr, rr);
            tc::mul2(y0, y1, y0, y1, nw[j], nw[j + 1]);
            tc::mul2(y0, y1, y0, y1, sigmoid_fast(__uint_as_float(gw[e] << 16)),
                     sigmoid_fast(__uint_as_float(gw[e] & 0xffff0000u)));
            yw[e] = tc::bf16x2_rn(y0, y1);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(p.out + (size_t)(start + t0 + t) * HC + h * kDv + col0 + cofs);
        dst[part] = make_uint4(yw[0], yw[1], yw[2], yw[3]);
    };
    float o_pend[kHalfCols];   // the outputs and gate of the chunk sent last, finished next
    uint4 g_pend[2];
    float o_cur[kHalfCols], rr_prev = 0.f;
    put_state();
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    cluster_wait();
    // tensor memory (each product in two 32-column halves that add up to it, see
    // mma_split3_bcat): [W S; Qtil S (+ Aqk Ut)] alternates between columns 0 and 64 from chunk
    // to chunk, so that a chunk's outputs are read while the next chunk's first product runs;
    // Kbar^T Ut at column 128
    const uint32_t tmem = sm.tmem, d2 = tmem + 128;
    uint32_t ph_mma = 0, ph_a1 = 0, ph_rest = 0;   // ph_rest: bit bf = phase of rest buffer bf
    // what has been started and not yet waited for (bit 0: the [W; Qtil] copy, 1: a product,
    // 2 + bf: the copies into rest buffer bf); if a wait gives up, thread 0 waits for these
    // (bounded) before the tensor memory is freed and the CTA exits
    uint32_t pending = 1u | 4u;
    bool ok = true;

    for (int c = 0; c < nc && ok; c++) {
        const int t0 = c * C, n = L - t0 < C ? L - t0 : C;
        const int cb = c & 1;            // this chunk's buffer of K = tokens operands
        ScanRest &rs = sm.rest[cb];
        const uint32_t d1 = tmem + 64 * cb;
        // (S^T is in b1: written before the loop or by the previous chunk's update, then fenced
        // for the tensor core and followed by a barrier; [W; Qtil] has arrived: waited for here
        // for the first chunk, at the previous chunk's last barrier for the others)
        if (c == 0) {
            if (!(ok = wait_all(&sm.bar_a1, ph_a1, p.err_word))) break;
            ph_a1 ^= 1;
            pending &= ~1u;
        }
        if (tid == 0) {
            tc::mma_split3_bcat(d1, smem_u32(sm.a1[0]), smem_u32(sm.a1[1]), 128, smem_u32(sm.b1), kScanCols, 8, false);
            tc::commit(&sm.bar_mma);
        }
        // the next chunk's K = tokens operands into the other buffer (free since the previous
        // chunk's last barrier), issued by another warp while the product runs: issuing copies
        // takes the issuing thread a while, and thread 0 issues the products
        if (tid == 32 && c + 1 < nc) issue_rest(c + 1, cb ^ 1);
        pending |= 2u | (c + 1 < nc ? 4u << (cb ^ 1) : 0u);
        // the previous chunk's outputs, from the other accumulator, meanwhile (the next product
        // into that accumulator follows the fenced barriers of this chunk): chunk c - 2's sums
        // read, chunk c - 1's sent; chunk c - 2 is finished half while the Ut operand is built,
        // half while the second product runs
        if (quarter >= 2 && c > 0) {
            ld_cat(tc::taddr(tmem + 64 * (cb ^ 1), 32 * quarter, cofs), o_cur);
            rr_prev = c > 1 ? norm_read(c - 2) : 0.f;
            norm_send(c - 1, o_cur);
        }
        // the first product and this chunk's K = tokens operands, one synchronisation for both
        if (!(ok = wait_all2(&sm.bar_mma, ph_mma, &sm.bar_rest[cb], (ph_rest >> cb) & 1u, p.err_word))) break;
        ph_mma ^= 1;
        ph_rest ^= 1u << cb;
        pending &= ~(2u | (4u << cb));
        // [W; Qtil] has been consumed: the next chunk's copy is issued by a warp that has no
        // part in the Ut operand
        if (tid == 64 && c + 1 < nc) issue_a1(c + 1);
        if (c + 1 < nc) pending |= 1u;
        // Ut = U - W S as the B operand (MN-major: N = 32 columns, K = 64 tokens): the warps of
        // lane quarters 0, 1 hold token t = row's row of W S and write their 16 columns of it
        if (quarter < 2) {
            const int t = row;
            float x[kHalfCols];
            ld_cat(tc::taddr(d1, 32 * quarter, cofs), x);
            const float *ur = &rs.u[t][0];
#pragma unroll
            for (int g = 0; g < kHalfCols / 4; g++) {
                const float4 u4 = ld4(ur + (((cofs / 4 + g) ^ (t & 7)) << 2));
                tc::sub2(x[4 * g], x[4 * g + 1], u4.x, u4.y, x[4 * g], x[4 * g + 1]);
                tc::sub2(x[4 * g + 2], x[4 * g + 3], u4.z, u4.w, x[4 * g + 2], x[4 * g + 3]);
                if (t >= n) x[4 * g] = x[4 * g + 1] = x[4 * g + 2] = x[4 * g + 3] = 0.f;
            }
#pragma unroll
            for (int g = 0; g < kHalfCols / 8; g++) put_cat(sm.b2, cofs + 8 * g, t, &x[8 * g]);
        } else if (c > 1) {
            norm_finish(c - 2, o_pend, g_pend, rr_prev, 0);
        }
        tc::fence_smem_to_async();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (tid == 0) {
            // Kbar^T Ut -> d2;  [0; Aqk] Ut accumulated onto [W S; Qtil S] -> rows 64.. = O
            tc::mma_split3_bcat(d2, smem_u32(rs.a2[0]), smem_u32(rs.a2[1]), C, smem_u32(sm.b2), kScanCols, 4, false);
            tc::mma_split3_bcat(d1, smem_u32(rs.aqk[0]) - C * C * 2, smem_u32(rs.aqk[1]) - C * C * 2, C, smem_u32(sm.b2),
                                kScanCols, 4, true);
            tc::commit(&sm.bar_mma);
        }
        pending |= 2u;
        // the rest of chunk c - 2 finished while the second product runs (registers and global
        // memory only)
        if (quarter >= 2 && c > 0) {
            if (c > 1) norm_finish(c - 2, o_pend, g_pend, rr_prev, 1);
            load_gate(c - 1, g_pend);
#pragma unroll
            for (int j = 0; j < kHalfCols; j++) o_pend[j] = o_cur[j];
        }
        if (!(ok = wait_all(&sm.bar_mma, ph_mma, p.err_word))) break;
        ph_mma ^= 1;
        pending &= ~2u;
        {
            float ds[kHalfCols];
            ld_cat(tc::taddr(d2, 32 * quarter, cofs), ds);
            const float dcay = rs.d[row];
#pragma unroll
            for (int j = 0; j < kHalfCols; j += 2) tc::fma2(S[j], S[j + 1], dcay, dcay, S[j], S[j + 1], ds[j], ds[j + 1]);
            put_state();   // the next chunk's S^T (this chunk's first product has completed)
        }
        tc::fence_smem_to_async();   // the next chunk's S^T, for the tensor core
        tc::fence_before_sync();
        // this chunk's buffer (u, d, Kbar^T, Aqk) is no longer read; the next chunk's [W; Qtil]
        // is waited for in the same synchronisation
        if (c + 1 < nc) {
            if (!(ok = wait_all(&sm.bar_a1, ph_a1, p.err_word))) break;
            ph_a1 ^= 1;
            pending &= ~1u;
        } else {
            __syncthreads();
            tc::fence_after_sync();
        }
    }
    // the last chunk's outputs: finish the one before, send the last's sums, finish it
    if (ok && quarter >= 2) {
        float o[kHalfCols];
        uint4 g[2];
        ld_cat(tc::taddr(tmem + 64 * ((nc - 1) & 1), 32 * quarter, cofs), o);
        const float rr = nc > 1 ? norm_read(nc - 2) : 0.f;
        norm_send(nc - 1, o);
        if (nc > 1) {
            norm_finish(nc - 2, o_pend, g_pend, rr, 0);
            norm_finish(nc - 2, o_pend, g_pend, rr, 1);
        }
        load_gate(nc - 1, g);
        const float rr_last = norm_read(nc - 1);
        norm_finish(nc - 1, o, g, rr_last, 0);
        norm_finish(nc - 1, o, g, rr_last, 1);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();   // the deallocation follows every warp's tensor-memory loads
    if (!ok && tid == 0) {
        if (pending & 1u) mbar_wait_bounded(&sm.bar_a1, ph_a1, kWaitLimitNs);
        if (pending & 2u) mbar_wait_bounded(&sm.bar_mma, ph_mma, kWaitLimitNs);
        for (int bf = 0; bf < 2; bf++)
            if (pending & (4u << bf)) mbar_wait_bounded(&sm.bar_rest[bf], (ph_rest >> bf) & 1u, kWaitLimitNs);
    }
    tc::fence_before_sync();
    __syncthreads();   // on the error path, thread 0 has waited for what was in flight
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, kScanTmemCols);
    // no CTA leaves while another may still write its sums into it
    cluster_arrive();
    cluster_wait();
    if (!ok) return;
    // final state (one rounding to the storage dtype)
#pragma unroll
    for (int j = 0; j < kHalfCols; j++) tile[(size_t)row * kDv + col0 + cofs + j] = (ST)S[j];
    // final conv window of the head's channels: z = [window, x_0 .. x_{L-1}], keep z[L .. L+2]
    if (blk == 0) {
        for (int it = tid; it < 3 * kDk; it += NTB) {
            const int tens = it / kDk, ch = h * kDk + it % kDk;
            const __nv_bfloat16 *src = tens == 0 ? p.q : tens == 1 ? p.k : p.v;
            __nv_bfloat16 w[3];
            for (int j = 0; j < 3; j++) {
                const int zi = L + j;   // index into z
                w[j] = zi < 3 ? p.conv_state[(((size_t)slot * 3 + tens) * kTaps + zi) * HC + ch]
                              : src[(size_t)(start + zi - 3) * HC + ch];
            }
            for (int j = 0; j < 3; j++) p.conv_state[(((size_t)slot * 3 + tens) * kTaps + j) * HC + ch] = w[j];
        }
    }
}

}  // namespace

size_t prefill_workspace_bytes(int H, int B, int L)
{
    if (H <= 0 || B <= 0 || L <= 0) return 0;
    const size_t n_chunks = (size_t)(L + C - 1) / C;
    return (size_t)B * H * n_chunks * kRecBytes;
}

size_t prefill_varlen_workspace_bytes(int H, int B, long total_tokens)
{
    if (H <= 0 || B <= 0 || total_tokens <= 0) return 0;
    return ((size_t)total_tokens / C + (size_t)B) * H * kRecBytes;
}

// The scan as clusters of the kScanBlocks column-block CTAs of a (sequence, head).
template <typename Kern>
cudaError_t launch_scan(Kern kern, dim3 grid, cudaStream_t stream, const RecurrentParams &p, const uint8_t *ws, int n_chunks)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(NTB);
    cfg.dynamicSmemBytes = sizeof(ScanSmem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kScanBlocks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, ws, n_chunks);
}

cudaError_t launch_prefill(const RecurrentParams &p, bool bf16_state, void *workspace, cudaStream_t stream)
{
    static KernelSetup setup_prep, setup_scan_f, setup_scan_b;
    const int n_chunks = (p.T + C - 1) / C;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    cudaError_t e = setup_prep.get(kda_chunk_prep, NTA, sizeof(PrepSmem), 0, nullptr);
    if (e != cudaSuccess) return e;
    kda_chunk_prep<<<dim3((unsigned)n_chunks, (unsigned)p.H, (unsigned)p.B), NTA, sizeof(PrepSmem), stream>>>(p, ws, n_chunks);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const dim3 sgrid(kScanBlocks, (unsigned)p.H, (unsigned)p.B);
    if (bf16_state) {
        if ((e = setup_scan_b.get(kda_chunk_scan<__nv_bfloat16>, NTB, sizeof(ScanSmem), 0, nullptr)) != cudaSuccess) return e;
        return launch_scan(kda_chunk_scan<__nv_bfloat16>, sgrid, stream, p, ws, n_chunks);
    }
    if ((e = setup_scan_f.get(kda_chunk_scan<float>, NTB, sizeof(ScanSmem), 0, nullptr)) != cudaSuccess) return e;
    return launch_scan(kda_chunk_scan<float>, sgrid, stream, p, ws, n_chunks);
}

}  // namespace kda
