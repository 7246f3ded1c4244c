// kda_tile.cu -- the token-serial KDA mixer step: single-token decode and multi-token draft
// verify, each optionally resuming from the previous step's records (the commit fused in).
//
// One CTA of 256 threads owns one (sequence, head) tile: the 128 x 128 recurrent state of that
// head, held in FP32 registers for the whole launch whatever the storage dtype.  Two CTAs share
// an SM.  Launches are programmatic dependent launches; the CTA's critical path is kept to the
// unavoidable memory round trips:
//   - before the dependency wait, warp 0 starts bulk async copies (TMA) of the layer's weights
//     (the head's W_fb rows, 32 KiB, and dt_bias) into shared memory, every thread loads its
//     conv channels' weights (kept packed until the conv), and one thread starts an L2
//     prefetch of the state tile the slot id names at that moment (a hint only);
//   - after it, warp 0 copies the pre-conv q, k, v, gate rows and f_a of up to 16 tokens, all
//     completing on one mbarrier, while every thread reads the slot id and issues its 128-bit
//     loads of the state tile (a warp covers one 512-byte FP32 row or two 256-byte BF16 rows
//     per instruction) and of its conv-window channels.
// Then, per group of up to 16 tokens, the gates of all its tokens are computed at once ("KDA
// fuses the f_b projection, convolution, FP32 recurrence and gated output normalization",
// NVFP4 Kimi K3 targets page, Description):
//   f_b projection: a half-warp owns 8 W rows, a lane 8 of the 128 f_a entries of each; the 8
//     independent partial dot products are combined by a butterfly reduce-scatter over the
//     16 lanes (8 shuffles in all) -> alpha = exp(g);
//   short causal conv + SiLU of the head's q, k, v channels (window in registers);
//   |q|^2, |k|^2, q.k (warp reductions) and beta;
// and token by token, on the register tile:
//   S <- Diag(alpha) S with S^T k and S^T q in the same sweep (cross-warp reduction in smem),
//   u = v - S^T k, o = S^T q + beta u (k.q) = (updated S)^T q, gated RMSNorm of o,
//   S += beta k u^T.
// Verify ("FP32 per-token draft records with either SSM storage dtype", same page; per-token
// KDA verify states, Kimi K3 on modeling_v2 page, section 5) writes the FP32 state and the conv
// window after every token and leaves the slot untouched (or, resuming, commits the starting
// record to it); decode writes the final state (rounded once to the storage dtype) and window
// back to the slot.  Further down, with the same arithmetic: kda_decode_kernel serves
// single-token decode of BF16 pools at four CTAs per SM, kda_decode_pair_kernel single-token
// decode of FP32 pools with two tiles per CTA when one tile per CTA would take more than a wave,
// kda_decode_cluster_kernel single-token decode of few tiles, each split over a cluster of four
// CTAs.  Every kernel has an instance for FP8 E4M3 projection weights with per-row scales (the
// scale multiplies each finished f_b dot product).
#include <cstddef>

#include "kda_internal.cuh"
#include "kda_ptx.cuh"

namespace kda {
namespace {

constexpr int NT = 256;
constexpr int kGroup = 16;                            // tokens whose gates are computed together
constexpr uint64_t kWaitLimitNs = 2000000000ull;      // no wait of this kernel spins longer than 2 s
constexpr int kRowBytes = 128 * 2;                    // one head's channels of a bf16 row
constexpr int kHeadBytes = kDk * kRank * 2 + kDk * 4; // W_fb rows + dt_bias of one head
constexpr int kFp8HeadBytes = kDk * kRank + kDk * 4 + kDk * 4;   // FP8 codes + row scales + dt_bias

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float softplusf_(float x) { return x > 20.0f ? x : log1pf(expf(x)); }
// The verify forms' gates (which equal the decode results to FP32 rounding only, their f_b
// projection being summed on the tensor cores) use the fast exponential, logarithm and divide
// (errors of a few ulp); decode keeps the full-precision forms above.
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }
__device__ __forceinline__ float softplus_fast(float x) { return x > 20.0f ? x : __logf(1.0f + __expf(x)); }

// Packed FP32 arithmetic: two lanes per instruction, each lane an IEEE round-to-nearest
// operation, so the results equal the scalar fmaf / multiply bit for bit.
__device__ __forceinline__ void fma2(float &d0, float &d1, float a0, float a1, float b0, float b1, float c0, float c1)
{
    asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void mul2(float &d0, float &d1, float a0, float a1, float b0, float b1)
{
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

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

__device__ __forceinline__ void unpack8(const uint4 &r, float *f)
{
    f[0] = bf16_lo(r.x); f[1] = bf16_hi(r.x); f[2] = bf16_lo(r.y); f[3] = bf16_hi(r.y);
    f[4] = bf16_lo(r.z); f[5] = bf16_hi(r.z); f[6] = bf16_lo(r.w); f[7] = bf16_hi(r.w);
}

// W_fb row `row` of head h, entries [8 li, 8 li + 8), as floats, read through L1: BF16
// weights, or FP8 E4M3 codes (exact; the row's scale is applied to the finished dot product).
template <bool W8>
__device__ __forceinline__ void load_w8(const RecurrentParams &p, int h, int row, int li, float *w)
{
    const size_t off = ((size_t)h * kDk + row) * kRank + li * 8;
    if constexpr (W8) e4m3x8_to_f32(__ldg(reinterpret_cast<const uint2 *>(p.W_fb8 + off)), w);
    else unpack8(__ldg(reinterpret_cast<const uint4 *>(p.W_fb + off)), w);
}

// A finished f_b dot product of row `row` of head h times that row's FP8 scale (BF16: as is).
template <bool W8>
__device__ __forceinline__ float row_scaled(const RecurrentParams &p, int h, int row, float v)
{
    if constexpr (W8) return v * __ldg(p.W_fb_scale + (size_t)h * kDk + row);
    else return v;
}

// ---- f_b projection of the verify forms on the tensor cores
//
// alpha[t][r] = sum_k W_fb[h dk + r][k] f_a[t][k] for the 128 rows r of head h and up to 8
// tokens t per chain of warp-level MMAs (m16n8k16, BF16 operands, FP32 accumulation); warp w
// owns rows [16 w, 16 w + 16).  Lane (g, c) = (lane / 4, lane % 4) holds, for each block of 32
// k, the 8 consecutive entries [32 blk + 8 c, 32 blk + 8 c + 8) of rows 16 w + g and
// 16 w + g + 8 (A) and of token g (B): the block's first MMA takes entries 0..3 of every lane's
// 8, the second entries 4..7, so each k position of the MMA pairs the same W and f_a entry and
// every product enters the sum once.  The chain runs the blocks in order from zero, so a
// (row, token) gets the same bits in every verify launch.  E4M3 codes convert to BF16 exactly;
// the row's FP8 scale multiplies the finished sum.  A verify group of T tokens takes 8 MMAs per
// warp instead of T x (64 FMAs, 64 unpacks, 8 shuffles) per thread.  Single-token decode keeps
// the FMA chain of the decode kernels (measured on GB300: with the MMA chain those kernels wait
// on its latency and slow down by 1 to 5 %), so verify outputs and records equal the decode
// results to FP32 rounding rather than bit for bit.
__device__ __forceinline__ void mma_16816(float *d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 8 E4M3 codes as 8 BF16 values (exact: every E4M3 value is a BF16 value)
__device__ __forceinline__ uint4 e4m3x8_to_bf16(uint2 v)
{
    float f[8];
    e4m3x8_to_f32(v, f);
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

// The chain for n <= 8 tokens whose f_a rows are fa(t) (the other columns zero).  wa(i, blk)
// gives the lane's entries of row 16 w + g + 8 i in block blk.  Afterwards d[j] (j = 0, 1) is
// row 16 w + g, token 2 c + j, and d[2 + j] row 16 w + g + 8, token 2 c + j.
template <typename WA, typename FA>
__device__ __forceinline__ void fb_chain(WA wa, FA fa, int n, int lane, float *d)
{
    const int g = lane >> 2, c = lane & 3;
    d[0] = d[1] = d[2] = d[3] = 0.f;
    const __nv_bfloat16 *frow = g < n ? fa(g) : nullptr;
#pragma unroll
    for (int blk = 0; blk < 4; blk++) {
        const uint4 f = frow ? *reinterpret_cast<const uint4 *>(frow + 32 * blk + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
        const uint4 w0 = wa(0, blk), w1 = wa(1, blk);
        mma_16816(d, w0.x, w1.x, w0.y, w1.y, f.x, f.y);
        mma_16816(d, w0.z, w1.z, w0.w, w1.w, f.z, f.w);
    }
}

// Hands the chain's sums to put(t, row, v) for the tokens t < n.
template <typename PUT>
__device__ __forceinline__ void fb_put(const float *d, int warp, int lane, int n, PUT put)
{
    const int r = 16 * warp + (lane >> 2), t = 2 * (lane & 3);
#pragma unroll
    for (int i = 0; i < 2; i++) {
#pragma unroll
        for (int j = 0; j < 2; j++)
            if (t + j < n) put(t + j, r + 8 * i, d[2 * i + j]);
    }
}

// Register tile: a thread owns columns [col, col+VEC) of rows row0 + RPP*p, p < NP.
template <typename ST>
struct Tile {
    static constexpr int VEC = 16 / sizeof(ST);   // 4 (fp32) or 8 (bf16) columns per thread
    static constexpr int TPR = kDv / VEC;          // threads per row: 32 or 16
    static constexpr int RPP = NT / TPR;           // rows per pass: 8 or 16
    static constexpr int NP = kDk / RPP;           // passes: 16 or 8
};

__device__ __forceinline__ void unpack(const uint4 &r, float *f, float)
{
    f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
}

__device__ __forceinline__ void unpack(const uint4 &r, float *f, __nv_bfloat16) { unpack8(r, f); }

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

// Shared memory: [ head: W bf16 [128][128], dt_bias f32 [128]
//                | staged inputs bf16: q, k, v, gate [G][128] each, f_a [G][128]
//                | gate arrays f32 [G][128]: alpha (f_b sums first), q, k, v after the conv;
//                  per token |q|^2, |k|^2, q.k, beta
//                | fixed ]
struct __align__(16) Fixed {
    alignas(16) float red[NT / 32][2][kDv];   // per-warp partial S^T k / S^T q
    alignas(16) float u[kDv];
    alignas(16) float norm_w[kDv];
    alignas(16) float rms[4];
    alignas(8) uint64_t in_bar;               // W, dt_bias and the group's inputs
};
static_assert(offsetof(Fixed, red) % 16 == 0 && offsetof(Fixed, u) % 16 == 0 &&
              offsetof(Fixed, norm_w) % 16 == 0 && offsetof(Fixed, in_bar) % 8 == 0,
              "shared-memory alignment");
static_assert(kHeadBytes % 128 == 0, "staging alignment");

__host__ __device__ constexpr size_t staged_off() { return (size_t)kHeadBytes; }
__host__ __device__ constexpr size_t gate_off(int G) { return staged_off() + (size_t)5 * G * kRowBytes; }
__host__ __device__ constexpr size_t fixed_off(int G) { return (gate_off(G) + (size_t)G * (4 * 128 + 4) * 4 + 15) & ~(size_t)15; }
__host__ __device__ constexpr size_t smem_total(int G) { return fixed_off(G) + sizeof(Fixed); }

// While the previous kernel on the stream drains: an L2 prefetch of the state tile (and, with
// `window`, the conv window) sequence b will read, chosen from its slot id (and accepted length,
// when resuming) as they read at this moment.  The reads go to L2 (no copy that could turn
// stale stays in L1) and are bounds-checked; the outcome is only a hint.  The kernel loads the
// tile and window from the values it reads after the dependency wait.  (Measured on GB300: the
// window rows pay off for multi-token verify, not for single-token decode.)
template <typename ST>
__device__ __forceinline__ void prefetch_before_wait(const RecurrentParams &p, int b, int h, bool window)
{
    const int H = p.H, HC = H * kDk;
    if (p.prev_accepted) {
        const int na = __ldcg(p.prev_accepted + b);
        if (na > 0 && na <= p.prev_T) {
            const size_t rt = (size_t)b * p.prev_T + na - 1;
            bulk_prefetch_l2(p.prev_rec_state + (rt * H + h) * (kDk * kDv), kDk * kDv * 4);
            for (int r = 0; window && r < 3 * kTaps; r++)
                bulk_prefetch_l2(p.prev_rec_conv + (rt * 3 * kTaps + r) * HC + (size_t)h * kDk, kRowBytes);
            return;
        }
    }
    const int s = __ldcg(p.slot_ids + b);
    if (s < 0 || s >= p.num_slots) return;
    bulk_prefetch_l2(reinterpret_cast<const ST *>(p.state) + ((size_t)s * H + h) * (kDk * kDv), kDk * kDv * sizeof(ST));
    for (int r = 0; window && r < 3 * kTaps; r++)
        bulk_prefetch_l2(p.conv_state + ((size_t)s * 3 * kTaps + r) * HC + (size_t)h * kDk, kRowBytes);
}

// Only the first resident wave of CTAs can start while the previous kernel on the stream is
// still running; a later CTA starts after one of this launch's CTAs has exited, so for it the
// previous kernel has finished and a speculative prefetch would only add a round trip to its
// start.
__device__ __forceinline__ bool first_wave(const RecurrentParams &p)
{
    return p.prefetch_stride <= 0 || (long)blockIdx.y * gridDim.x + blockIdx.x < (long)p.prefetch_stride;
}

// L2 prefetch of the per-token inputs of (sequence b, head h): the q, k, v and gate rows and the
// f_a rows of its first n tokens (a hint, like the state-tile prefetch).
__device__ __forceinline__ void prefetch_inputs_l2(const RecurrentParams &p, int b, int h, int n)
{
    const size_t HC = (size_t)p.H * kDk, tok0 = (size_t)b * p.T;
    for (int t = 0; t < n; t++) {
        const size_t off = (tok0 + t) * HC + (size_t)h * kDk;
        bulk_prefetch_l2(p.q + off, kRowBytes);
        bulk_prefetch_l2(p.k + off, kRowBytes);
        bulk_prefetch_l2(p.v + off, kRowBytes);
        bulk_prefetch_l2(p.gate + off, kRowBytes);
    }
    bulk_prefetch_l2(p.f_a + tok0 * kRank, (uint32_t)n * kRowBytes);
}

// One conv channel a thread owns: which of q, k, v, its channel, and its window (the three
// previous pre-conv inputs).  The channel's taps are held packed beside it (two BF16 per word).
struct ConvItem {
    int tensor, ch;
    __nv_bfloat16 win[kTaps];
};

template <typename ST, bool RECORDS, bool W8>
__global__ void __launch_bounds__(NT, 2) kda_tile_kernel(const RecurrentParams p)
{
    using TL = Tile<ST>;
    constexpr int VEC = TL::VEC, TPR = TL::TPR, RPP = TL::RPP, NP = TL::NP;
    extern __shared__ __align__(128) uint8_t smem[];
    const int T = p.T, G = T < kGroup ? T : kGroup;
    const __nv_bfloat16 *Wh = reinterpret_cast<const __nv_bfloat16 *>(smem);
    const float *dtb = reinterpret_cast<const float *>(smem + kDk * kRank * 2);
    const __nv_bfloat16 *xs = reinterpret_cast<const __nv_bfloat16 *>(smem + staged_off());   // [4][G][128]
    const __nv_bfloat16 *fas = xs + 4 * G * 128;                                             // [G][128]
    float *g_alpha = reinterpret_cast<float *>(smem + gate_off(G));
    float *g_q = g_alpha + G * kDk, *g_k = g_q + G * kDk, *g_v = g_k + G * kDk, *g_nrm = g_v + G * kDv;
    Fixed &fx = *reinterpret_cast<Fixed *>(smem + fixed_off(G));

    const int h = blockIdx.x, b = blockIdx.y, H = p.H, HC = H * kDk;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // warp 0: stage the inputs of tokens [g0, g0 + n) into shared memory, completing on
    // fx.in_bar; `expect` registers their bytes (the first group's are registered together with
    // the head's W_fb rows and dt_bias, which are copied before the grid dependency wait)
    auto issue_inputs = [&](int g0, int n, bool expect) {
        if (expect && lane == 0) mbar_arrive_expect_tx(&fx.in_bar, (uint32_t)(5 * n) * kRowBytes);
        __syncwarp();
        const size_t tok0 = (size_t)b * T + g0;
        for (int c = lane; c < 4 * n + 1; c += 32) {
            if (c < 4 * n) {
                const int which = c / n, t = c % n;
                const __nv_bfloat16 *base = which == 0 ? p.q : which == 1 ? p.k : which == 2 ? p.v : p.gate;
                bulk_load(smem + staged_off() + ((size_t)which * G + t) * kRowBytes,
                          base + (tok0 + t) * HC + (size_t)h * kDk, kRowBytes, &fx.in_bar);
            } else {
                bulk_load(smem + staged_off() + (size_t)4 * G * kRowBytes, p.f_a + tok0 * kRank,
                          (uint32_t)n * kRowBytes, &fx.in_bar);
            }
        }
    };
    // all threads: wait for the staged inputs (bounded); false when the wait gave up
    uint32_t in_phase = 0;
    auto inputs_arrived = [&]() -> bool {
        const bool ok = mbar_wait_bounded(&fx.in_bar, in_phase, kWaitLimitNs);
        in_phase ^= 1u;
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicOr(p.err_word, KDA_DEVERR_TIMEOUT);
                mbar_wait_bounded(&fx.in_bar, in_phase ^ 1u, kWaitLimitNs);
            }
            return false;
        }
        return true;
    };

    // ---- 1. the layer's weights (written by no kernel) may be read before the previous kernel
    //      on the stream has finished; everything else is read for use only after
    //      grid_dependency_wait() (before it, one thread reads the slot id, and the accepted
    //      length when resuming, speculatively, only to aim an L2 prefetch)
    // (norm_w is held in a register and stored after the slot id's load has been issued: a
    // shared-memory store here would wait for its load before the dependency wait)
    const float nw = tid < kDv ? __ldg(p.norm_w + tid) : 0.f;
    const float a_log = __ldg(p.A_log + h);
    // conv items: item 0 = q channel tid (tid < 128) or k channel tid - 128; item 1 = v channel
    // tid.  Their weights are layer weights: loaded here, unpacked where the conv uses them.
    const int n_items = tid < kDv ? 2 : 1;
    uint2 cwr[2];
#pragma unroll
    for (int it = 0; it < 2; it++) {
        const int tens = it == 0 ? (tid < kDk ? 0 : 1) : 2;
        if (it < n_items) cwr[it] = __ldg(reinterpret_cast<const uint2 *>(p.conv_w + ((size_t)tens * HC + h * kDk + (tid & (kDk - 1))) * kConv));
    }
    constexpr bool fp8 = W8;   // FP8 E4M3 weights with per-row scales
    if (warp == 0) {
        if (lane == 0) {
            mbar_init(&fx.in_bar, 1);
            fence_mbar_init();
            mbar_arrive_expect_tx(&fx.in_bar, (fp8 ? kFp8HeadBytes : kHeadBytes) + (uint32_t)(5 * G) * kRowBytes);
        }
        __syncwarp();
        // BF16: W rows at 0, dt_bias at 32 KiB; FP8: codes at 0, row scales at 16 KiB
        if (lane == 0) {
            if constexpr (fp8) bulk_load(smem, p.W_fb8 + (size_t)h * kDk * kRank, kDk * kRank, &fx.in_bar);
            else bulk_load(smem, p.W_fb + (size_t)h * kDk * kRank, kDk * kRank * 2, &fx.in_bar);
        }
        if (lane == 1) bulk_load(smem + kDk * kRank * 2, p.dt_bias + (size_t)h * kDk, kDk * 4, &fx.in_bar);
        if (lane == 2 && fp8) bulk_load(smem + kDk * kRank, p.W_fb_scale + (size_t)h * kDk, kDk * 4, &fx.in_bar);
        grid_dependency_wait();
        issue_inputs(0, G, false);
    } else {
        if (tid == 32) prefetch_before_wait<ST>(p, b, h, RECORDS);
        grid_dependency_wait();
    }
    // ---- 2. slot id, then the slot's state tile and conv window
    const int slot = __ldg(p.slot_ids + b);
    if (tid < kDv) fx.norm_w[tid] = nw;
    const float a_h = expf(a_log);
    __syncthreads();   // fx.in_bar is initialised before anyone waits on it
    if (slot < 0 || slot >= p.num_slots) {
        // nothing to compute; the copies already started must land before the CTA exits
        if (tid == 0) {
            atomicOr(p.err_word, KDA_DEVERR_SLOT);
            mbar_wait_bounded(&fx.in_bar, 0, kWaitLimitNs);
        }
        return;
    }
    // resume: the previous step's accepted length n picks the starting point, record n - 1 of
    // the previous step's records (n >= 1) or the slot (n = 0)
    int n_prev = 0;
    if (p.prev_accepted) {
        n_prev = __ldg(p.prev_accepted + b);
        if (n_prev < 0 || n_prev > p.prev_T) {
            if (tid == 0) {
                atomicOr(p.err_word, KDA_DEVERR_ACCEPTED);
                mbar_wait_bounded(&fx.in_bar, 0, kWaitLimitNs);
            }
            return;
        }
    }
    const int Tb = p.n_tokens ? __ldg(p.n_tokens + b) : T;   // tokens of this sequence
    const int col = (tid % TPR) * VEC, row0 = tid / TPR;
    ST *tile = reinterpret_cast<ST *>(p.state) + ((size_t)slot * H + h) * (kDk * kDv);
    const float *rec0 = n_prev > 0 ? p.prev_rec_state + (((size_t)b * p.prev_T + n_prev - 1) * H + h) * (kDk * kDv) : nullptr;
    const __nv_bfloat16 *win0 = n_prev > 0 ? p.prev_rec_conv + ((size_t)b * p.prev_T + n_prev - 1) * 3 * kTaps * HC
                                           : p.conv_state + (size_t)slot * 3 * kTaps * HC;
    // The CTA that takes this CTA's place one wave later works on item (b * H + h) +
    // prefetch_stride: pull its state tile and conv window into L2 ahead of time, so that its
    // first memory round trip after the slot id is an L2 hit.  Issued at the start when the
    // launch has many waves, after this CTA's own gates otherwise (so it does not compete with
    // the first wave's loads).
    auto prefetch_next_wave = [&]() {
        if (tid != 32 || p.prefetch_stride <= 0) return;
        const long nxt = (long)b * H + h + p.prefetch_stride;
        if (nxt >= (long)p.B * H) return;
        const int nb = (int)(nxt / H), nh = (int)(nxt % H);
        const int na = p.prev_accepted ? __ldg(p.prev_accepted + nb) : 0;
        if (na > 0 && na <= p.prev_T) {
            const size_t rt = (size_t)nb * p.prev_T + na - 1;
            bulk_prefetch_l2(p.prev_rec_state + (rt * H + nh) * (kDk * kDv), kDk * kDv * 4);
            for (int r = 0; r < 3 * kTaps; r++)
                bulk_prefetch_l2(p.prev_rec_conv + (rt * 3 * kTaps + r) * HC + (size_t)nh * kDk, kRowBytes);
            return;
        }
        const int ns = __ldg(p.slot_ids + nb);
        if (ns < 0 || ns >= p.num_slots) return;
        bulk_prefetch_l2(reinterpret_cast<const ST *>(p.state) + ((size_t)ns * H + nh) * (kDk * kDv),
                         kDk * kDv * sizeof(ST));
        for (int r = 0; r < 3 * kTaps; r++)
            bulk_prefetch_l2(p.conv_state + ((size_t)ns * 3 * kTaps + r) * HC + (size_t)nh * kDk, kRowBytes);
    };
    if (p.prefetch_early) prefetch_next_wave();
    float st[NP][VEC];
    uint4 raw[sizeof(ST) == 2 ? NP : 1];   // BF16 tiles land packed and are unpacked after the gates
    if (rec0) {
        // FP32 record: BF16 tiles are rounded to storage after the gates, as a commit stores them
#pragma unroll
        for (int pp = 0; pp < NP; pp++) {
#pragma unroll
            for (int c = 0; c < VEC; c += 4) {
                const float4 r = __ldcs(reinterpret_cast<const float4 *>(rec0 + (size_t)(row0 + RPP * pp) * kDv + col + c));
                st[pp][c] = r.x; st[pp][c + 1] = r.y; st[pp][c + 2] = r.z; st[pp][c + 3] = r.w;
            }
        }
    } else {
#pragma unroll
        for (int pp = 0; pp < NP; pp++) {
            const uint4 r = __ldcs(reinterpret_cast<const uint4 *>(tile + (size_t)(row0 + RPP * pp) * kDv + col));
            if constexpr (sizeof(ST) == 4) unpack(r, st[pp], ST());
            else raw[pp] = r;
        }
    }
    // conv items: item 0 = q channel tid (tid < 128) or k channel tid - 128; item 1 = v channel tid
    ConvItem cv[2];
#pragma unroll
    for (int it = 0; it < 2; it++) {
        if (it < n_items) {
            cv[it].tensor = it == 0 ? (tid < kDk ? 0 : 1) : 2;
            cv[it].ch = h * kDk + (tid & (kDk - 1));
#pragma unroll
            for (int j = 0; j < kTaps; j++)
                cv[it].win[j] = win0[((size_t)cv[it].tensor * kTaps + j) * HC + cv[it].ch];
        }
    }
    const float q_scale = rsqrtf((float)kDk);

    // Gates of tokens [g0, g0 + n) from the staged inputs: f_b projection, conv, norms, beta.
    auto gate_group = [&](int g0, int n) {
        const size_t tok0 = (size_t)b * T + g0;
        // beta stays packed until the sigmoid, so no thread waits for it before the projection
        const __nv_bfloat16 bt = tid < n ? p.beta[(tok0 + tid) * H + h] : __nv_bfloat16();
        // a1, verify: the f_b projection of the group's tokens on the tensor cores, 8 tokens per
        //     chain, from the head's W rows in shared memory
        if constexpr (RECORDS) {
            const uint8_t *W8h = smem;                                          // FP8 codes
            const float *w8s = reinterpret_cast<const float *>(smem + kDk * kRank);   // FP8 row scales
            auto wa = [&](int i, int blk) -> uint4 {
                const int off = (16 * warp + (lane >> 2) + 8 * i) * kRank + 32 * blk + 8 * (lane & 3);
                if constexpr (fp8) return e4m3x8_to_bf16(*reinterpret_cast<const uint2 *>(W8h + off));
                else return *reinterpret_cast<const uint4 *>(Wh + off);
            };
            for (int t0 = 0; t0 < n; t0 += 8) {
                const int m = n - t0 < 8 ? n - t0 : 8;
                float d[4];
                fb_chain(wa, [&](int t) { return fas + (t0 + t) * kRank; }, m, lane, d);
                fb_put(d, warp, lane, m, [&](int t, int row, float v) {
                    g_alpha[(t0 + t) * kDk + row] = fp8 ? v * w8s[row] : v;
                });
            }
        }
        // a1, decode: half-warp hw owns W rows 8 hw + j (j < 8); lane li owns f_a entries
        //     [8 li, 8 li + 8) (the FMA chain of the decode kernels)
        else {
            const int hw = tid >> 4, li = tid & 15;
            const int b3 = (li >> 3) & 1, b2 = (li >> 2) & 1, b1 = (li >> 1) & 1;
            const uint8_t *W8h = smem;                                          // FP8 codes
            const float *w8s = reinterpret_cast<const float *>(smem + kDk * kRank);   // FP8 row scales
            for (int t = 0; t < n; t++) {
                float f[8];
                unpack8(*reinterpret_cast<const uint4 *>(fas + t * kRank + li * 8), f);
                float acc[8];
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    float w[8];
                    if constexpr (fp8) e4m3x8_to_f32(*reinterpret_cast<const uint2 *>(W8h + (hw * 8 + j) * kRank + li * 8), w);
                    else unpack8(*reinterpret_cast<const uint4 *>(Wh + (hw * 8 + j) * kRank + li * 8), w);
                    float a = w[0] * f[0];
#pragma unroll
                    for (int e = 1; e < 8; e++) a = fmaf(w[e], f[e], a);
                    acc[j] = a;
                }
                // butterfly reduce-scatter over the 16 lanes: afterwards lanes li and li^1 hold
                // the full sum of row 8 hw + (4 b3 + 2 b2 + b1)
                float v4[4], v2[2];
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const float keep = b3 ? acc[j + 4] : acc[j], give = b3 ? acc[j] : acc[j + 4];
                    v4[j] = keep + __shfl_xor_sync(0xffffffffu, give, 8);
                }
#pragma unroll
                for (int j = 0; j < 2; j++) {
                    const float keep = b2 ? v4[j + 2] : v4[j], give = b2 ? v4[j] : v4[j + 2];
                    v2[j] = keep + __shfl_xor_sync(0xffffffffu, give, 4);
                }
                float v1 = (b1 ? v2[1] : v2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? v2[0] : v2[1], 2);
                v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
                const int row = hw * 8 + 4 * b3 + 2 * b2 + b1;
                if ((li & 1) == 0) g_alpha[t * kDk + row] = fp8 ? v1 * w8s[row] : v1;
            }
        }
        // a4: conv + SiLU over the staged inputs; window shift; verify records the window
#pragma unroll
        for (int it = 0; it < 2; it++) {
            if (it < n_items) {
                const int tens = cv[it].tensor, ch = cv[it].ch, c = ch - h * kDk;
                float *dst = tens == 0 ? g_q : (tens == 1 ? g_k : g_v);
                for (int t = 0; t < n; t++) {
                    const __nv_bfloat16 x = xs[(tens * G + t) * kDk + c];
                    float acc = bf16_lo(cwr[it].x) * bf2f(cv[it].win[0]);
                    acc = fmaf(bf16_hi(cwr[it].x), bf2f(cv[it].win[1]), acc);
                    acc = fmaf(bf16_lo(cwr[it].y), bf2f(cv[it].win[2]), acc);
                    acc = fmaf(bf16_hi(cwr[it].y), bf2f(x), acc);
                    dst[t * kDk + c] = RECORDS ? silu_fast(acc) : acc / (1.0f + expf(-acc));
                    cv[it].win[0] = cv[it].win[1];
                    cv[it].win[1] = cv[it].win[2];
                    cv[it].win[2] = x;
                    if (RECORDS) {
#pragma unroll
                        for (int j = 0; j < kTaps; j++)
                            p.rec_conv[(((tok0 + t) * 3 + tens) * kTaps + j) * HC + ch] = cv[it].win[j];
                    }
                }
            }
        }
        __syncthreads();
        // a2 decay, a5 norms and q.k, a3 beta
        for (int i = tid; i < n * kDk; i += NT)
            g_alpha[i] = RECORDS ? __expf(-a_h * softplus_fast(g_alpha[i] + dtb[i & (kDk - 1)]))
                                 : expf(-a_h * softplusf_(g_alpha[i] + dtb[i & (kDk - 1)]));
        for (int pr = warp; pr < 3 * n; pr += NT / 32) {
            const int t = pr / 3, kind = pr % 3;
            const float *a = (kind == 1 ? g_k : g_q) + t * kDk;
            const float *c = (kind == 0 ? g_q : g_k) + t * kDk;
            const float4 x = *reinterpret_cast<const float4 *>(a + lane * 4);
            const float4 y = *reinterpret_cast<const float4 *>(c + lane * 4);
            float sum = x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
            sum = group_sum<32>(sum);
            if (lane == 0) g_nrm[t * 4 + kind] = sum;
        }
        if (tid < n) g_nrm[tid * 4 + 3] = sigmoidf_(bf2f(bt));
        __syncthreads();
    };

    // Tokens [g0, g0 + n) on the register tile.
    auto token_group = [&](int g0, int n) {
        const size_t tok0 = (size_t)b * T + g0;
        for (int t = 0; t < n; t++) {
            const size_t tok = tok0 + t;
            const float *nrm = g_nrm + t * 4;
            const float rq = q_scale / sqrtf(nrm[0] + p.l2_eps);
            const float rk = 1.0f / sqrtf(nrm[1] + p.l2_eps);
            const float kq = nrm[2] * rq * rk;
            const float beta = nrm[3];
            const float *al = g_alpha + t * kDk, *kv = g_k + t * kDk, *qv = g_q + t * kDk;

            // a6: decay + S^T k, S^T q
            float ak[VEC], aq[VEC];
#pragma unroll
            for (int c = 0; c < VEC; c++) ak[c] = aq[c] = 0.f;
#pragma unroll
            for (int pp = 0; pp < NP; pp++) {
                const int i = row0 + RPP * pp;
                const float a = al[i], akk = a * (kv[i] * rk), aqq = a * (qv[i] * rq);
#pragma unroll
                for (int c = 0; c < VEC; c++) {
                    const float s0 = st[pp][c];
                    st[pp][c] = s0 * a;
                    ak[c] = fmaf(s0, akk, ak[c]);
                    aq[c] = fmaf(s0, aqq, aq[c]);
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
            // u, o, RMS partials
            float o = 0.f;
            if (tid < kDv) {
                float stk = 0.f, stq = 0.f;
#pragma unroll
                for (int w = 0; w < NT / 32; w++) { stk += fx.red[w][0][tid]; stq += fx.red[w][1][tid]; }
                const float u = g_v[t * kDv + tid] - stk;
                o = stq + beta * u * kq;
                fx.u[tid] = u;
                const float ss = group_sum<32>(o * o);
                if (lane == 0) fx.rms[warp] = ss;
            }
            __syncthreads();
            if (tid < kDv) {
                const float ms = (fx.rms[0] + fx.rms[1] + fx.rms[2] + fx.rms[3]) * (1.0f / kDv);
                const size_t oi = tok * (size_t)(H * kDv) + (size_t)h * kDv + tid;
                const float gt = bf2f(xs[(3 * G + t) * kDv + tid]);
                const float y = o * rsqrtf(ms + p.norm_eps) * fx.norm_w[tid] * sigmoidf_(gt);
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
            // no barrier before the next token: its writes of fx.red, fx.u and fx.rms come after
            // its first barrier, which every reader of this token's values reaches only after
            // reading them
        }
    };

    // verify resume: commit the starting record to the slot (the window now, the state below)
    auto commit_window = [&]() {
#pragma unroll
        for (int it = 0; it < 2; it++) {
            if (it < n_items) {
#pragma unroll
                for (int j = 0; j < kTaps; j++)
                    p.conv_state[(((size_t)slot * 3 + cv[it].tensor) * kTaps + j) * HC + cv[it].ch] = cv[it].win[j];
            }
        }
    };
    auto commit_state = [&]() {
#pragma unroll
        for (int pp = 0; pp < NP; pp++)
            __stcs(reinterpret_cast<uint4 *>(tile + (size_t)(row0 + RPP * pp) * kDv + col), pack(st[pp], ST()));
    };
    auto round_to_storage = [&]() {   // BF16 tile started from an FP32 record
        if constexpr (sizeof(ST) == 2) {
#pragma unroll
            for (int pp = 0; pp < NP; pp++)
#pragma unroll
                for (int c = 0; c < VEC; c++) st[pp][c] = __bfloat162float(__float2bfloat16_rn(st[pp][c]));
        }
    };
    if (RECORDS && rec0) commit_window();
    if (Tb < 1 || Tb > T) {
        if (RECORDS && rec0) {
            round_to_storage();
            commit_state();
        }
        if (tid == 0) {
            atomicOr(p.err_word, KDA_DEVERR_TOKENS);
            mbar_wait_bounded(&fx.in_bar, 0, kWaitLimitNs);
        }
        return;
    }
    const int G0 = Tb < G ? Tb : G;
    if (!inputs_arrived()) return;
    gate_group(0, G0);
    if (!p.prefetch_early) prefetch_next_wave();
    if (rec0) {
        round_to_storage();
        if (RECORDS) commit_state();
    } else if constexpr (sizeof(ST) == 2) {
#pragma unroll
        for (int pp = 0; pp < NP; pp++) unpack(raw[pp], st[pp], ST());
    }
    token_group(0, G0);
    for (int g0 = G; g0 < Tb; g0 += G) {
        const int n = Tb - g0 < G ? Tb - g0 : G;
        __syncthreads();   // the previous group's readers of the staged inputs and gates are done
        if (warp == 0) issue_inputs(g0, n, true);
        if (!inputs_arrived()) return;
        gate_group(g0, n);
        token_group(g0, n);
    }

    if (!RECORDS) {
        // the state, rounded once to the storage dtype, and the conv window go back to the slot
#pragma unroll
        for (int pp = 0; pp < NP; pp++)
            __stcs(reinterpret_cast<uint4 *>(tile + (size_t)(row0 + RPP * pp) * kDv + col), pack(st[pp], ST()));
#pragma unroll
        for (int it = 0; it < 2; it++) {
            if (it < n_items) {
#pragma unroll
                for (int j = 0; j < kTaps; j++)
                    p.conv_state[(((size_t)slot * 3 + cv[it].tensor) * kTaps + j) * HC + cv[it].ch] = cv[it].win[j];
            }
        }
    }
}

// ============================================================================ decode
//
// Single-token decode of a BF16 pool with a smaller per-CTA footprint, so that four CTAs share
// an SM: the tile lives in shared memory (one 32 KiB bulk async copy, so no registers are tied
// up by the loads in flight); W_fb rows are read through L1 / L2.  Two sweeps over the tile:
// decay with S^T k and S^T q, then decay again with the rank-1 update and the store.  Each thread reads the same
// elements and sums them in the same order as kda_tile_kernel, so a decode here equals the
// tile kernel's decode bit for bit.  (Measured on GB300, 256 x 32 BF16 tiles: 125 us per launch
// with the shared-memory tile at four CTAs per SM, 145 us with it packed in registers at three.)
struct __align__(16) DecodeFixed {
    alignas(16) float red[NT / 32][2][kDv];
    alignas(16) float u[kDv];
    alignas(16) float norm_w[kDv];
    alignas(16) float alpha[kDk];
    alignas(16) float q[kDk];
    alignas(16) float k[kDk];
    alignas(16) float v[kDv];
    alignas(16) float nrm[4];
    alignas(16) float rms[4];
    alignas(16) __nv_bfloat16 xs[5][128];   // staged q, k, v, gate rows and f_a
    alignas(16) float dtb[kDk];
    alignas(8) uint64_t in_bar, tile_bar;
};

// The whole tile in shared memory: 32 KiB, brought in by one bulk async copy.
template <typename ST>
__host__ __device__ constexpr size_t decode_tile_smem() { return (size_t)kDk * kDv * sizeof(ST); }

template <typename ST>
__host__ __device__ constexpr size_t decode_smem() { return decode_tile_smem<ST>() + sizeof(DecodeFixed); }

// Four CTAs per SM (register budget 65536 / (256 x 4)).
template <typename ST, bool W8>
__global__ void __launch_bounds__(NT, 4) kda_decode_kernel(const RecurrentParams p)
{
    static_assert(sizeof(ST) == 2, "single-token decode of BF16 pools (FP32 pools run the tile and paired kernels)");
    using TL = Tile<ST>;
    constexpr int VEC = TL::VEC, TPR = TL::TPR, RPP = TL::RPP, NP = TL::NP;
    constexpr uint32_t SBYTES = (uint32_t)decode_tile_smem<ST>();
    static_assert(SBYTES % 16 == 0, "bulk copy size");
    extern __shared__ __align__(128) uint8_t smem[];
    const ST *tile_s = reinterpret_cast<const ST *>(smem);
    DecodeFixed &fx = *reinterpret_cast<DecodeFixed *>(smem + decode_tile_smem<ST>());

    const int h = blockIdx.x, b = blockIdx.y, H = p.H, HC = H * kDk;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // ---- 1. the layer's weights (dt_bias, W_fb towards L2, norm_w, A_log) before the wait for
    //      the previous kernel on the stream; the token's rows and everything else after it
    // (held in registers and stored after the slot id's load has been issued: a shared-memory
    // store here would wait for its load before the dependency wait, on the start of every CTA
    // after the first wave)
    const float nw = tid < kDv ? __ldg(p.norm_w + tid) : 0.f;
    const float a_log = __ldg(p.A_log + h);
    // conv items: item 0 = q channel tid (tid < 128) or k channel tid - 128; item 1 = v channel
    // tid.  Their weights are layer weights: loaded here, unpacked where the conv uses them.
    const int n_items = tid < kDv ? 2 : 1;
    uint2 cwr[2];
#pragma unroll
    for (int it = 0; it < 2; it++) {
        const int tens = it == 0 ? (tid < kDk ? 0 : 1) : 2;
        if (it < n_items) cwr[it] = __ldg(reinterpret_cast<const uint2 *>(p.conv_w + ((size_t)tens * HC + h * kDk + (tid & (kDk - 1))) * kConv));
    }
    if (warp == 0) {
        if (lane == 0) {
            mbar_init(&fx.in_bar, 1);
            mbar_init(&fx.tile_bar, 1);
            fence_mbar_init();
            mbar_arrive_expect_tx(&fx.in_bar, 5 * kRowBytes + kDk * 4);
        }
        __syncwarp();
        if (lane == 5) bulk_load(fx.dtb, p.dt_bias + (size_t)h * kDk, kDk * 4, &fx.in_bar);
        if (lane == 6) {
            if constexpr (W8) bulk_prefetch_l2(p.W_fb8 + (size_t)h * kDk * kRank, kDk * kRank);
            else bulk_prefetch_l2(p.W_fb + (size_t)h * kDk * kRank, kDk * kRank * 2);
        }
        grid_dependency_wait();
        if (lane < 4) {
            const __nv_bfloat16 *base = lane == 0 ? p.q : lane == 1 ? p.k : lane == 2 ? p.v : p.gate;
            bulk_load(fx.xs[lane], base + (size_t)b * HC + (size_t)h * kDk, kRowBytes, &fx.in_bar);
        } else if (lane == 4) {
            bulk_load(fx.xs[4], p.f_a + (size_t)b * kRank, kRowBytes, &fx.in_bar);
        }
    } else {
        if (tid == 32 && first_wave(p)) prefetch_before_wait<ST>(p, b, h, false);
        grid_dependency_wait();
    }
    // ---- 2. slot id, then the slot's tile and conv window
    const int slot = __ldg(p.slot_ids + b);
    if (tid < kDv) fx.norm_w[tid] = nw;
    const float a_h = expf(a_log);
    __syncthreads();   // the mbarriers are initialised before anyone waits on them
    if (slot < 0 || slot >= p.num_slots) {
        if (tid == 0) {
            atomicOr(p.err_word, KDA_DEVERR_SLOT);
            mbar_wait_bounded(&fx.in_bar, 0, kWaitLimitNs);
        }
        return;
    }
    ST *tile = reinterpret_cast<ST *>(p.state) + ((size_t)slot * H + h) * (kDk * kDv);
    if (tid == 0) {
        mbar_arrive_expect_tx(&fx.tile_bar, SBYTES);
        bulk_load(smem, tile, SBYTES, &fx.tile_bar);
    }
    const int col = (tid % TPR) * VEC, row0 = tid / TPR;
    // the CTA that takes this CTA's place one wave later: its inputs, tile and window into L2,
    // after this CTA's gates (its slot id is read now, so that nothing waits for it then)
    const long nxt = (long)b * H + h + p.prefetch_stride;
    const bool has_next = tid == 32 && p.prefetch_stride > 0 && nxt < (long)p.B * H;
    const int nb = (int)(nxt / H), nh = (int)(nxt % H);
    const int ns = has_next ? __ldg(p.slot_ids + nb) : -1;
    ConvItem cv[2];
#pragma unroll
    for (int it = 0; it < 2; it++) {
        if (it < n_items) {
            cv[it].tensor = it == 0 ? (tid < kDk ? 0 : 1) : 2;
            cv[it].ch = h * kDk + (tid & (kDk - 1));
#pragma unroll
            for (int j = 0; j < kTaps; j++)
                cv[it].win[j] = p.conv_state[(((size_t)slot * 3 + cv[it].tensor) * kTaps + j) * HC + cv[it].ch];
        }
    }
    const __nv_bfloat16 braw = tid == 224 ? p.beta[(size_t)b * H + h] : __nv_bfloat16();   // converted where used

    // ---- 3. gates
    {
        const bool ok = mbar_wait_bounded(&fx.in_bar, 0, kWaitLimitNs);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicOr(p.err_word, KDA_DEVERR_TIMEOUT);
                mbar_wait_bounded(&fx.in_bar, 0, kWaitLimitNs);
                mbar_wait_bounded(&fx.tile_bar, 0, kWaitLimitNs);
            }
            return;
        }
    }
    // a1: half-warp hw owns W rows 8 hw + j; lane li owns f_a entries [8 li, 8 li + 8)
    {
        const int hw = tid >> 4, li = tid & 15;
        const int b3 = (li >> 3) & 1, b2 = (li >> 2) & 1, b1 = (li >> 1) & 1;
        float f[8];
        unpack8(*reinterpret_cast<const uint4 *>(&fx.xs[4][li * 8]), f);
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; j++) {
            float w[8];
            load_w8<W8>(p, h, hw * 8 + j, li, w);
            float a = w[0] * f[0];
#pragma unroll
            for (int e = 1; e < 8; e++) a = fmaf(w[e], f[e], a);
            acc[j] = a;
        }
        float v4[4], v2[2];
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const float keep = b3 ? acc[j + 4] : acc[j], give = b3 ? acc[j] : acc[j + 4];
            v4[j] = keep + __shfl_xor_sync(0xffffffffu, give, 8);
        }
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const float keep = b2 ? v4[j + 2] : v4[j], give = b2 ? v4[j] : v4[j + 2];
            v2[j] = keep + __shfl_xor_sync(0xffffffffu, give, 4);
        }
        float v1 = (b1 ? v2[1] : v2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? v2[0] : v2[1], 2);
        v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
        const int row = hw * 8 + 4 * b3 + 2 * b2 + b1;
        if ((li & 1) == 0) fx.alpha[row] = row_scaled<W8>(p, h, row, v1);
    }
    // a4: conv + SiLU, window shift
#pragma unroll
    for (int it = 0; it < 2; it++) {
        if (it < n_items) {
            const int tens = cv[it].tensor, c = cv[it].ch - h * kDk;
            float *dst = tens == 0 ? fx.q : (tens == 1 ? fx.k : fx.v);
            const __nv_bfloat16 x = fx.xs[tens][c];
            float acc = bf16_lo(cwr[it].x) * bf2f(cv[it].win[0]);
            acc = fmaf(bf16_hi(cwr[it].x), bf2f(cv[it].win[1]), acc);
            acc = fmaf(bf16_lo(cwr[it].y), bf2f(cv[it].win[2]), acc);
            acc = fmaf(bf16_hi(cwr[it].y), bf2f(x), acc);
            dst[c] = acc / (1.0f + expf(-acc));
            cv[it].win[0] = cv[it].win[1];
            cv[it].win[1] = cv[it].win[2];
            cv[it].win[2] = x;
        }
    }
    __syncthreads();
    // a2 decay, a5 norms and q.k, a3 beta
    if (tid < kDk) fx.alpha[tid] = expf(-a_h * softplusf_(fx.alpha[tid] + fx.dtb[tid]));
    if (warp >= 4 && warp < 7) {
        const int kind = warp - 4;
        const float *a = kind == 1 ? fx.k : fx.q;
        const float *c = kind == 0 ? fx.q : fx.k;
        const float4 x = *reinterpret_cast<const float4 *>(a + lane * 4);
        const float4 y = *reinterpret_cast<const float4 *>(c + lane * 4);
        float sum = x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
        sum = group_sum<32>(sum);
        if (lane == 0) fx.nrm[kind] = sum;
    }
    if (tid == 224) fx.nrm[3] = sigmoidf_(bf2f(braw));
    // the gates are written; the tile is waited for in the same synchronisation
    {
        const bool ok = mbar_wait_bounded(&fx.tile_bar, 0, kWaitLimitNs);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicOr(p.err_word, KDA_DEVERR_TIMEOUT);
                mbar_wait_bounded(&fx.tile_bar, 0, kWaitLimitNs);
            }
            return;
        }
    }
    if (has_next) {
        prefetch_inputs_l2(p, nb, nh, 1);
        if (ns >= 0 && ns < p.num_slots) {
            bulk_prefetch_l2(reinterpret_cast<const ST *>(p.state) + ((size_t)ns * H + nh) * (kDk * kDv),
                             kDk * kDv * sizeof(ST));
            for (int r = 0; r < 3 * kTaps; r++)
                bulk_prefetch_l2(p.conv_state + ((size_t)ns * 3 * kTaps + r) * HC + (size_t)nh * kDk, kRowBytes);
        }
    }

    // ---- 4. the sweeps
    const float rq = rsqrtf((float)kDk) / sqrtf(fx.nrm[0] + p.l2_eps);
    const float rk = 1.0f / sqrtf(fx.nrm[1] + p.l2_eps);
    const float kq = fx.nrm[2] * rq * rk;
    const float beta = fx.nrm[3];
    auto row_vals = [&](int pp, float *sv) {
        unpack(*reinterpret_cast<const uint4 *>(tile_s + (size_t)(row0 + RPP * pp) * kDv + col), sv, ST());
    };
    float ak[VEC], aq[VEC];
#pragma unroll
    for (int c = 0; c < VEC; c++) ak[c] = aq[c] = 0.f;
#pragma unroll
    for (int pp = 0; pp < NP; pp++) {
        const int i = row0 + RPP * pp;
        float sv[VEC];
        row_vals(pp, sv);
        const float a = fx.alpha[i], akk = a * (fx.k[i] * rk), aqq = a * (fx.q[i] * rq);
        // packed FP32 (measured on GB300: 103.0 -> 98.9 us per launch on decode_b256; the
        // paired kernel, latency-bound, measured slower with it and keeps the scalar form)
#pragma unroll
        for (int c = 0; c < VEC; c += 2) {
            fma2(ak[c], ak[c + 1], sv[c], sv[c + 1], akk, akk, ak[c], ak[c + 1]);
            fma2(aq[c], aq[c + 1], sv[c], sv[c + 1], aqq, aqq, aq[c], aq[c + 1]);
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
    float o = 0.f;
    if (tid < kDv) {
        float stk = 0.f, stq = 0.f;
#pragma unroll
        for (int w = 0; w < NT / 32; w++) { stk += fx.red[w][0][tid]; stq += fx.red[w][1][tid]; }
        const float u = fx.v[tid] - stk;
        o = stq + beta * u * kq;
        fx.u[tid] = u;
        const float ss = group_sum<32>(o * o);
        if (lane == 0) fx.rms[warp] = ss;
    }
    __syncthreads();
    if (tid < kDv) {
        const float ms = (fx.rms[0] + fx.rms[1] + fx.rms[2] + fx.rms[3]) * (1.0f / kDv);
        const float y = o * rsqrtf(ms + p.norm_eps) * fx.norm_w[tid] * sigmoidf_(bf2f(fx.xs[3][tid]));
        p.out[(size_t)b * (H * kDv) + (size_t)h * kDv + tid] = __float2bfloat16_rn(y);
    }
    float uu[VEC];
#pragma unroll
    for (int c = 0; c < VEC; c += 4) {
        const float4 u4 = *reinterpret_cast<const float4 *>(&fx.u[col + c]);
        uu[c] = u4.x; uu[c + 1] = u4.y; uu[c + 2] = u4.z; uu[c + 3] = u4.w;
    }
#pragma unroll
    for (int pp = 0; pp < NP; pp++) {
        const int i = row0 + RPP * pp;
        float sv[VEC];
        row_vals(pp, sv);
        const float a = fx.alpha[i], bk = beta * fx.k[i] * rk;
#pragma unroll
        for (int c = 0; c < VEC; c += 2) {
            float m0, m1;
            mul2(m0, m1, sv[c], sv[c + 1], a, a);
            fma2(sv[c], sv[c + 1], bk, bk, uu[c], uu[c + 1], m0, m1);
        }
        __stcs(reinterpret_cast<uint4 *>(tile + (size_t)i * kDv + col), pack(sv, ST()));
    }
#pragma unroll
    for (int it = 0; it < 2; it++) {
        if (it < n_items) {
#pragma unroll
            for (int j = 0; j < kTaps; j++)
                p.conv_state[(((size_t)slot * 3 + cv[it].tensor) * kTaps + j) * HC + cv[it].ch] = cv[it].win[j];
        }
    }
}

// ============================================================================ paired decode
//
// Single-token decode of an FP32 pool (or decode resuming from the previous step's records) with
// two tiles per CTA, (2c, h) and (2c + 1, h), so that
// a launch of up to two resident waves of one-tile CTAs runs as one wave, and the second tile's
// work follows the first's on the same CTA instead of waiting for a free slot.  The first tile
// keeps rows 0..63 in registers and rows 64..127 in shared memory, the second lives in shared
// memory.  Order of the memory traffic: the first tile is prefetched into L2 before the
// dependency wait and loaded right after the slot ids, together with both tokens' inputs and
// windows; the second tile is copied only once the gates of both tiles are done (measured on
// GB300: earlier starts, or a pre-wait prefetch of it, slow the launch, because at the wait
// release they compete with what the first half of the chain needs).  The gates of both tiles
// are computed in one phase, then each tile's sweeps run back to back; each tile's gates and
// sweeps are those of kda_decode_kernel<float> (same elements per thread, same order of sums),
// so the result equals the tile kernel's decode bit for bit.
struct __align__(16) PairFixed {
    alignas(16) float red[NT / 32][2][kDv];
    alignas(16) float u[kDv];
    alignas(16) float norm_w[kDv];
    alignas(16) float alpha[2][kDk];          // per tile: the gates of its token
    alignas(16) float q[2][kDk];
    alignas(16) float k[2][kDk];
    alignas(16) float v[2][kDv];
    alignas(16) float nrm[2][4];
    alignas(16) float rms[4];
    alignas(16) __nv_bfloat16 xs[2][5][128];   // per tile: staged q, k, v, gate rows and f_a
    alignas(16) float dtb[kDk];
    alignas(8) uint64_t in_bar, tile_bar[2];
};

constexpr uint32_t kPairTileA = 64 * kDv * 4;    // rows 64..127 of the first tile
constexpr uint32_t kPairTileB = kDk * kDv * 4;   // the whole second tile
__host__ __device__ constexpr size_t pair_smem() { return (size_t)kPairTileA + kPairTileB + sizeof(PairFixed); }
// two CTAs per SM: 228 KiB of shared memory per SM, 1 KiB of it reserved per CTA
static_assert(2 * (pair_smem() + 1024) <= 228 * 1024, "two paired-decode CTAs per SM");

template <int J>
struct TileIx { static constexpr int value = J; };

template <bool W8, bool RESUME>
__global__ void __launch_bounds__(NT, 2) kda_decode_pair_kernel(const RecurrentParams p)
{
    using TL = Tile<float>;
    constexpr int VEC = TL::VEC, TPR = TL::TPR, RPP = TL::RPP, NP = TL::NP;
    constexpr int NREG = NP / 2;   // passes of the first tile held in registers (rows 0..63)
    extern __shared__ __align__(128) uint8_t smem[];
    const float *tsA = reinterpret_cast<const float *>(smem);
    const float *tsB = reinterpret_cast<const float *>(smem + kPairTileA);
    PairFixed &fx = *reinterpret_cast<PairFixed *>(smem + kPairTileA + kPairTileB);

    const int h = blockIdx.x, H = p.H, HC = H * kDk;
    const int b0 = 2 * (int)blockIdx.y;
    const int nt = b0 + 1 < p.B ? 2 : 1;   // tiles of this CTA
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // ---- 1. the layer's weights before the dependency wait, the tokens' rows after it
    if (tid < kDv) fx.norm_w[tid] = __ldg(p.norm_w + tid);
    const float a_h = expf(__ldg(p.A_log + h));
    // conv items: item 0 = q channel tid (tid < 128) or k channel tid - 128; item 1 = v channel
    // tid.  Their weights are layer weights: loaded here, unpacked where the conv uses them.
    const int n_items = tid < kDv ? 2 : 1;
    uint2 cwr[2];
#pragma unroll
    for (int it = 0; it < 2; it++) {
        const int tens = it == 0 ? (tid < kDk ? 0 : 1) : 2;
        if (it < n_items) cwr[it] = __ldg(reinterpret_cast<const uint2 *>(p.conv_w + ((size_t)tens * HC + h * kDk + (tid & (kDk - 1))) * kConv));
    }
    if (warp == 0) {
        if (lane == 0) {
            mbar_init(&fx.in_bar, 1);
            mbar_init(&fx.tile_bar[0], 1);
            mbar_init(&fx.tile_bar[1], 1);
            fence_mbar_init();
            mbar_arrive_expect_tx(&fx.in_bar, (uint32_t)(5 * nt) * kRowBytes + kDk * 4);
        }
        __syncwarp();
        if (lane == 5) bulk_load(fx.dtb, p.dt_bias + (size_t)h * kDk, kDk * 4, &fx.in_bar);
        if (lane == 6) {
            if constexpr (W8) bulk_prefetch_l2(p.W_fb8 + (size_t)h * kDk * kRank, kDk * kRank);
            else bulk_prefetch_l2(p.W_fb + (size_t)h * kDk * kRank, kDk * kRank * 2);
        }
        grid_dependency_wait();
        const int j = lane >> 3, r = lane & 7;   // lanes 0..4: the first token, 8..12: the second
        if (j < nt && r < 5) {
            const int bj = b0 + j;
            if (r < 4) {
                const __nv_bfloat16 *base = r == 0 ? p.q : r == 1 ? p.k : r == 2 ? p.v : p.gate;
                bulk_load(fx.xs[j][r], base + (size_t)bj * HC + (size_t)h * kDk, kRowBytes, &fx.in_bar);
            } else {
                bulk_load(fx.xs[j][4], p.f_a + (size_t)bj * kRank, kRowBytes, &fx.in_bar);
            }
        }
    } else {
        if (tid == 32) prefetch_before_wait<float>(p, b0, h, false);
        grid_dependency_wait();
    }
    // ---- 2. slot ids (and, resuming, the previous step's accepted lengths), then both tiles
    //      and conv windows
    const int s0 = __ldg(p.slot_ids + b0);
    const int s1 = nt == 2 ? __ldg(p.slot_ids + b0 + 1) : -1;
    int n0 = 0, n1 = 0;
    if constexpr (RESUME) {
        n0 = __ldg(p.prev_accepted + b0);
        n1 = nt == 2 ? __ldg(p.prev_accepted + b0 + 1) : 0;
    }
    __syncthreads();   // the mbarriers are initialised before anyone waits on them
    bool ok0 = s0 >= 0 && s0 < p.num_slots;
    bool ok1 = nt == 2 && s1 >= 0 && s1 < p.num_slots;
    if (tid == 0 && (!ok0 || (nt == 2 && !ok1))) atomicOr(p.err_word, KDA_DEVERR_SLOT);
    if constexpr (RESUME) {
        const bool acc0 = n0 >= 0 && n0 <= p.prev_T, acc1 = n1 >= 0 && n1 <= p.prev_T;
        if (tid == 0 && ((ok0 && !acc0) || (ok1 && !acc1))) atomicOr(p.err_word, KDA_DEVERR_ACCEPTED);
        ok0 = ok0 && acc0;
        ok1 = ok1 && acc1;
    }
    float *tile0 = reinterpret_cast<float *>(p.state) + ((size_t)(ok0 ? s0 : 0) * H + h) * (kDk * kDv);
    float *tile1 = reinterpret_cast<float *>(p.state) + ((size_t)(ok1 ? s1 : 0) * H + h) * (kDk * kDv);
    // resuming: where each tile starts, record n - 1 of the previous step (n >= 1) or the slot
    const float *src0 = tile0, *src1 = tile1;
    if constexpr (RESUME) {
        if (ok0 && n0 > 0) src0 = p.prev_rec_state + (((size_t)b0 * p.prev_T + n0 - 1) * H + h) * (kDk * kDv);
        if (ok1 && n1 > 0) src1 = p.prev_rec_state + (((size_t)(b0 + 1) * p.prev_T + n1 - 1) * H + h) * (kDk * kDv);
    }
    // the second tile's copy starts once the first tile's gates are done (so that the memory
    // system serves the first tile, the inputs and the windows first), or now if there is no
    // first tile; only thread 0 issues and drains copies
    bool issued1 = false;
    auto issue_tile1 = [&]() {
        if (tid == 0 && ok1 && !issued1) {
            mbar_arrive_expect_tx(&fx.tile_bar[1], kPairTileB);
            bulk_load(smem + kPairTileA, src1, kPairTileB, &fx.tile_bar[1]);
            issued1 = true;
        }
    };
    if (tid == 0) {
        if (ok0) {
            mbar_arrive_expect_tx(&fx.tile_bar[0], kPairTileA);
            bulk_load(smem, src0 + 64 * kDv, kPairTileA, &fx.tile_bar[0]);
        }
    }
    if (!ok0) issue_tile1();
    // every copy this CTA started lands before it exits, whatever happens below
    auto drain = [&]() {
        if (tid == 0) {
            mbar_wait_bounded(&fx.in_bar, 0, kWaitLimitNs);
            if (ok0) mbar_wait_bounded(&fx.tile_bar[0], 0, kWaitLimitNs);
            if (issued1) mbar_wait_bounded(&fx.tile_bar[1], 0, kWaitLimitNs);
        }
    };
    if (!ok0 && !ok1) {
        drain();
        return;
    }
    const int col = (tid % TPR) * VEC, row0 = tid / TPR;
    uint4 raw[NREG];
    if (ok0) {
#pragma unroll
        for (int pp = 0; pp < NREG; pp++)
            raw[pp] = __ldcs(reinterpret_cast<const uint4 *>(src0 + (size_t)(row0 + RPP * pp) * kDv + col));
    }
    // conv windows: one per tile (the weights are the same for both: same head)
    ConvItem cv[2];
    __nv_bfloat16 win1[2][kTaps];
#pragma unroll
    for (int it = 0; it < 2; it++) {
        if (it < n_items) {
            cv[it].tensor = it == 0 ? (tid < kDk ? 0 : 1) : 2;
            cv[it].ch = h * kDk + (tid & (kDk - 1));
#pragma unroll
            for (int t = 0; t < kTaps; t++) {
                if constexpr (RESUME) {
                    if (ok0) {
                        const __nv_bfloat16 *w0 = n0 > 0 ? p.prev_rec_conv + ((size_t)b0 * p.prev_T + n0 - 1) * 3 * kTaps * HC
                                                         : p.conv_state + (size_t)s0 * 3 * kTaps * HC;
                        cv[it].win[t] = w0[((size_t)cv[it].tensor * kTaps + t) * HC + cv[it].ch];
                    }
                    if (ok1) {
                        const __nv_bfloat16 *w1 = n1 > 0 ? p.prev_rec_conv + ((size_t)(b0 + 1) * p.prev_T + n1 - 1) * 3 * kTaps * HC
                                                         : p.conv_state + (size_t)s1 * 3 * kTaps * HC;
                        win1[it][t] = w1[((size_t)cv[it].tensor * kTaps + t) * HC + cv[it].ch];
                    }
                } else {
                    if (ok0) cv[it].win[t] = p.conv_state[(((size_t)s0 * 3 + cv[it].tensor) * kTaps + t) * HC + cv[it].ch];
                    if (ok1) win1[it][t] = p.conv_state[(((size_t)s1 * 3 + cv[it].tensor) * kTaps + t) * HC + cv[it].ch];
                }
            }
        }
    }
    __nv_bfloat16 braw[2] = {};   // converted where used, so no thread waits for them here
    if (tid == 224) {
        braw[0] = p.beta[(size_t)b0 * H + h];
        if (nt == 2) braw[1] = p.beta[(size_t)(b0 + 1) * H + h];
    }
    {
        const bool ok = mbar_wait_bounded(&fx.in_bar, 0, kWaitLimitNs);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) atomicOr(p.err_word, KDA_DEVERR_TIMEOUT);
            drain();
            return;
        }
    }

    // ---- 3. the gates of both tiles in one phase (f_b projection and conv per tile; then the
    //      decay of tile 0 on threads 0..127 and of tile 1 on 128..255, the norms of tile 0 on
    //      warps 4..6 and of tile 1 on warps 1..3), then each tile's sweeps
    // a1, resume instance: the f_b projection of both tiles' tokens (the tiles share the head):
    //     half-warp hw owns W rows 8 hw + i, lane li f_a entries [8 li, 8 li + 8); each W row is
    //     read and unpacked once and enters both tokens' dot products, each summed in the order
    //     of the other decode kernels (a second tile's row is not read when the CTA has one
    //     tile).  Measured on GB300: steady decode_resume 14.05 -> 13.63 us; the plain instance
    //     was 1 % slower this way and projects per tile below.
    if constexpr (RESUME) {
        const int hw = tid >> 4, li = tid & 15;
        const int b3 = (li >> 3) & 1, b2 = (li >> 2) & 1, b1 = (li >> 1) & 1;
        float f[2][8];
#pragma unroll
        for (int j = 0; j < 2; j++) {
            if (j < nt) unpack8(*reinterpret_cast<const uint4 *>(&fx.xs[j][4][li * 8]), f[j]);
            else for (int e = 0; e < 8; e++) f[j][e] = 0.f;
        }
        float acc[2][8];
#pragma unroll
        for (int i = 0; i < 8; i++) {
            float w[8];
            load_w8<W8>(p, h, hw * 8 + i, li, w);
#pragma unroll
            for (int j = 0; j < 2; j++) {
                float a = w[0] * f[j][0];
#pragma unroll
                for (int e = 1; e < 8; e++) a = fmaf(w[e], f[j][e], a);
                acc[j][i] = a;
            }
        }
#pragma unroll
        for (int j = 0; j < 2; j++) {
            float v4[4], v2[2];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const float keep = b3 ? acc[j][i + 4] : acc[j][i], give = b3 ? acc[j][i] : acc[j][i + 4];
                v4[i] = keep + __shfl_xor_sync(0xffffffffu, give, 8);
            }
#pragma unroll
            for (int i = 0; i < 2; i++) {
                const float keep = b2 ? v4[i + 2] : v4[i], give = b2 ? v4[i] : v4[i + 2];
                v2[i] = keep + __shfl_xor_sync(0xffffffffu, give, 4);
            }
            float v1 = (b1 ? v2[1] : v2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? v2[0] : v2[1], 2);
            v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
            const int row = hw * 8 + 4 * b3 + 2 * b2 + b1;
            if ((li & 1) == 0 && j < nt) fx.alpha[j][row] = row_scaled<W8>(p, h, row, v1);
        }
    }
    auto gates_a = [&](auto jt) {
        constexpr int j = decltype(jt)::value;
        // a1, plain instance: the tile's own projection (same sums)
        if constexpr (!RESUME) {
            const int hw = tid >> 4, li = tid & 15;
            const int b3 = (li >> 3) & 1, b2 = (li >> 2) & 1, b1 = (li >> 1) & 1;
            float f[8];
            unpack8(*reinterpret_cast<const uint4 *>(&fx.xs[j][4][li * 8]), f);
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; i++) {
                float w[8];
                load_w8<W8>(p, h, hw * 8 + i, li, w);
                float a = w[0] * f[0];
#pragma unroll
                for (int e = 1; e < 8; e++) a = fmaf(w[e], f[e], a);
                acc[i] = a;
            }
            float v4[4], v2[2];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const float keep = b3 ? acc[i + 4] : acc[i], give = b3 ? acc[i] : acc[i + 4];
                v4[i] = keep + __shfl_xor_sync(0xffffffffu, give, 8);
            }
#pragma unroll
            for (int i = 0; i < 2; i++) {
                const float keep = b2 ? v4[i + 2] : v4[i], give = b2 ? v4[i] : v4[i + 2];
                v2[i] = keep + __shfl_xor_sync(0xffffffffu, give, 4);
            }
            float v1 = (b1 ? v2[1] : v2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? v2[0] : v2[1], 2);
            v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
            const int row = hw * 8 + 4 * b3 + 2 * b2 + b1;
            if ((li & 1) == 0) fx.alpha[j][row] = row_scaled<W8>(p, h, row, v1);
        }
        // a4: conv + SiLU, window shift
#pragma unroll
        for (int it = 0; it < 2; it++) {
            if (it < n_items) {
                const ConvItem &c_ = cv[it];
                __nv_bfloat16 *win = j == 0 ? cv[it].win : win1[it];
                const int c = c_.ch - h * kDk;
                float *dst = c_.tensor == 0 ? fx.q[j] : (c_.tensor == 1 ? fx.k[j] : fx.v[j]);
                const __nv_bfloat16 x = fx.xs[j][c_.tensor][c];
                float acc = bf16_lo(cwr[it].x) * bf2f(win[0]);
                acc = fmaf(bf16_hi(cwr[it].x), bf2f(win[1]), acc);
                acc = fmaf(bf16_lo(cwr[it].y), bf2f(win[2]), acc);
                acc = fmaf(bf16_hi(cwr[it].y), bf2f(x), acc);
                dst[c] = acc / (1.0f + expf(-acc));
                win[0] = win[1];
                win[1] = win[2];
                win[2] = x;
            }
        }
    };
    if (ok0) gates_a(TileIx<0>{});
    if (ok1) gates_a(TileIx<1>{});
    __syncthreads();
    {
        const int j = tid >> 7, i = tid & (kDk - 1);
        if (j == 0 ? ok0 : ok1) fx.alpha[j][i] = expf(-a_h * softplusf_(fx.alpha[j][i] + fx.dtb[i]));
        const int nj = warp >= 4 ? 0 : 1, kind = warp >= 4 ? warp - 4 : warp - 1;
        if (warp != 0 && warp != 7 && (nj == 0 ? ok0 : ok1)) {
            const float *a = kind == 1 ? fx.k[nj] : fx.q[nj];
            const float *c = kind == 0 ? fx.q[nj] : fx.k[nj];
            const float4 x = *reinterpret_cast<const float4 *>(a + lane * 4);
            const float4 y = *reinterpret_cast<const float4 *>(c + lane * 4);
            float sum = x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
            sum = group_sum<32>(sum);
            if (lane == 0) fx.nrm[nj][kind] = sum;
        }
        if (tid == 224) {
            fx.nrm[0][3] = sigmoidf_(bf2f(braw[0]));
            fx.nrm[1][3] = sigmoidf_(bf2f(braw[1]));
        }
    }
    __syncthreads();
    issue_tile1();

    auto step = [&](auto jt) -> bool {
        constexpr int j = decltype(jt)::value;
        const int b = b0 + j;
        float *tile = j == 0 ? tile0 : tile1;
        // the sweeps
        const float rq = rsqrtf((float)kDk) / sqrtf(fx.nrm[j][0] + p.l2_eps);
        const float rk = 1.0f / sqrtf(fx.nrm[j][1] + p.l2_eps);
        const float kq = fx.nrm[j][2] * rq * rk;
        const float beta = fx.nrm[j][3];
        {
            const bool ok = mbar_wait_bounded(&fx.tile_bar[j], 0, kWaitLimitNs);
            if (__syncthreads_or(!ok)) return false;
        }
        auto row_vals = [&](int pp, float *sv) {
            if (j == 0 && pp < NREG) {
                unpack(raw[pp < NREG ? pp : 0], sv, float());
            } else {
                const float *ts = j == 0 ? tsA + (size_t)(row0 + RPP * pp - 64) * kDv : tsB + (size_t)(row0 + RPP * pp) * kDv;
                const float4 r = *reinterpret_cast<const float4 *>(ts + col);
                sv[0] = r.x; sv[1] = r.y; sv[2] = r.z; sv[3] = r.w;
            }
        };
        float ak[VEC], aq[VEC];
#pragma unroll
        for (int c = 0; c < VEC; c++) ak[c] = aq[c] = 0.f;
#pragma unroll
        for (int pp = 0; pp < NP; pp++) {
            const int i = row0 + RPP * pp;
            float sv[VEC];
            row_vals(pp, sv);
            const float a = fx.alpha[j][i], akk = a * (fx.k[j][i] * rk), aqq = a * (fx.q[j][i] * rq);
#pragma unroll
            for (int c = 0; c < VEC; c++) {
                ak[c] = fmaf(sv[c], akk, ak[c]);
                aq[c] = fmaf(sv[c], aqq, aq[c]);
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
        float o = 0.f;
        if (tid < kDv) {
            float stk = 0.f, stq = 0.f;
#pragma unroll
            for (int w = 0; w < NT / 32; w++) { stk += fx.red[w][0][tid]; stq += fx.red[w][1][tid]; }
            const float u = fx.v[j][tid] - stk;
            o = stq + beta * u * kq;
            fx.u[tid] = u;
            const float ss = group_sum<32>(o * o);
            if (lane == 0) fx.rms[warp] = ss;
        }
        __syncthreads();
        if (tid < kDv) {
            const float ms = (fx.rms[0] + fx.rms[1] + fx.rms[2] + fx.rms[3]) * (1.0f / kDv);
            const float y = o * rsqrtf(ms + p.norm_eps) * fx.norm_w[tid] * sigmoidf_(bf2f(fx.xs[j][3][tid]));
            p.out[(size_t)b * (H * kDv) + (size_t)h * kDv + tid] = __float2bfloat16_rn(y);
        }
        float uu[VEC];
#pragma unroll
        for (int c = 0; c < VEC; c += 4) {
            const float4 u4 = *reinterpret_cast<const float4 *>(&fx.u[col + c]);
            uu[c] = u4.x; uu[c + 1] = u4.y; uu[c + 2] = u4.z; uu[c + 3] = u4.w;
        }
#pragma unroll
        for (int pp = 0; pp < NP; pp++) {
            const int i = row0 + RPP * pp;
            float sv[VEC];
            row_vals(pp, sv);
            const float a = fx.alpha[j][i], bk = beta * fx.k[j][i] * rk;
#pragma unroll
            for (int c = 0; c < VEC; c++) sv[c] = fmaf(bk, uu[c], sv[c] * a);
            // a plain (write-back) store: measured 1 % faster here than a streaming one
            *reinterpret_cast<uint4 *>(tile + (size_t)i * kDv + col) = pack(sv, float());
        }
        const int sj = j == 0 ? s0 : s1;
#pragma unroll
        for (int it = 0; it < 2; it++) {
            if (it < n_items) {
                const __nv_bfloat16 *win = j == 0 ? cv[it].win : win1[it];
#pragma unroll
                for (int t = 0; t < kTaps; t++)
                    p.conv_state[(((size_t)sj * 3 + cv[it].tensor) * kTaps + t) * HC + cv[it].ch] = win[t];
            }
        }
        __syncthreads();   // fx.red, fx.u and fx.rms are reused by the next tile
        return true;
    };
    bool ok = true;
    if (ok0) ok = step(TileIx<0>{});
    if (ok && ok1) ok = step(TileIx<1>{});
    if (!ok) {
        if (tid == 0) atomicOr(p.err_word, KDA_DEVERR_TIMEOUT);
        drain();
    }
}

// ============================================================================ cluster decode
//
// Single-token decode when the B x H tiles would leave most SMs idle: each tile is split over a
// cluster of kClusterN CTAs, CTA rank c owning value columns [32 c, 32 c + 32) of the 128.  Every
// CTA computes the token's gates with the code of the decode kernels above (so the same values);
// a thread owns one column and the rows that the tile kernel's thread of that column owns, and
// sums them in the same order.  The one exchange is for the RMS norm: rank c sums o^2 over its
// 32 columns, the columns whose sum warp c of the tile kernel forms, in the same order, and
// writes that value into every CTA of the cluster through distributed shared memory; the state
// update and its stores overlap the exchange.  The result equals the tile kernel's decode bit
// for bit (so kda_decode_resume, which runs the tile kernel, still equals kda_commit +
// kda_decode).
constexpr int kClusterN = 4;
constexpr int kClusterCols = kDv / kClusterN;   // 32: one column per lane

struct __align__(16) ClusterFixed {
    alignas(16) float red[NT / 32][2][kClusterCols];   // per-warp partial S^T k / S^T q
    alignas(16) float u[kClusterCols];
    alignas(16) float norm_w[kDv];
    alignas(16) float alpha[kDk];
    alignas(16) float q[kDk];
    alignas(16) float k[kDk];
    alignas(16) float v[kDv];
    alignas(16) float nrm[4];
    alignas(16) float rms[4];
    alignas(16) __nv_bfloat16 xs[5][128];   // staged q, k, v, gate rows and f_a
    alignas(16) float dtb[kDk];
    alignas(8) uint64_t in_bar;
};

// Rows of the tile whose column-partial sums one thread of the tile kernel forms, in its order:
// FP32 tiles, warp w sums rows w + 8 pp (pp < 16); BF16 tiles, the two half-warps of warp w sum
// rows 2w + 16 pp and 2w + 1 + 16 pp (pp < 8), and the shuffle adds the second to the first.
template <typename ST>
__device__ __forceinline__ int cluster_row(int w, int e)
{
    if constexpr (sizeof(ST) == 4) return w + 8 * e;
    else return e < 8 ? 2 * w + 16 * e : 2 * w + 1 + 16 * (e - 8);
}

template <typename ST, bool W8>
__global__ void __launch_bounds__(NT) kda_decode_cluster_kernel(const RecurrentParams p)
{
    __shared__ ClusterFixed fx;
    const int h = blockIdx.x / kClusterN, b = blockIdx.y, H = p.H, HC = H * kDk;
    const int rank = (int)cluster_ctarank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int col = rank * kClusterCols + lane;   // this thread's column

    // every CTA of the cluster has started before any writes into another's shared memory
    cluster_arrive_relaxed();

    // ---- 1. the layer's weights before the dependency wait; the token's rows after it
    const float nw = tid < kDv ? __ldg(p.norm_w + tid) : 0.f;
    const float a_log = __ldg(p.A_log + h);
    const int n_items = tid < kDv ? 2 : 1;
    uint2 cwr[2];
#pragma unroll
    for (int it = 0; it < 2; it++) {
        const int tens = it == 0 ? (tid < kDk ? 0 : 1) : 2;
        if (it < n_items) cwr[it] = __ldg(reinterpret_cast<const uint2 *>(p.conv_w + ((size_t)tens * HC + h * kDk + (tid & (kDk - 1))) * kConv));
    }
    // this thread's W_fb entries (half-warp hw: rows 8 hw + j, lane li: entries 8 li ..), held in
    // registers from before the dependency wait: they are layer weights
    const int hw = tid >> 4, li = tid & 15;
    float wreg[8][8];
#pragma unroll
    for (int j = 0; j < 8; j++) load_w8<W8>(p, h, hw * 8 + j, li, wreg[j]);
    if (warp == 0) {
        if (lane == 0) {
            mbar_init(&fx.in_bar, 1);
            fence_mbar_init();
            mbar_arrive_expect_tx(&fx.in_bar, 5 * kRowBytes + kDk * 4);
        }
        __syncwarp();
        if (lane == 5) bulk_load(fx.dtb, p.dt_bias + (size_t)h * kDk, kDk * 4, &fx.in_bar);
        grid_dependency_wait();
        if (lane < 4) {
            const __nv_bfloat16 *base = lane == 0 ? p.q : lane == 1 ? p.k : lane == 2 ? p.v : p.gate;
            bulk_load(fx.xs[lane], base + (size_t)b * HC + (size_t)h * kDk, kRowBytes, &fx.in_bar);
        } else if (lane == 4) {
            bulk_load(fx.xs[4], p.f_a + (size_t)b * kRank, kRowBytes, &fx.in_bar);
        }
    } else {
        if (tid == 32 && rank == 0) prefetch_before_wait<ST>(p, b, h, false);
        grid_dependency_wait();
    }
    // ---- 2. slot id, then this CTA's columns of the tile and the conv window
    const int slot = __ldg(p.slot_ids + b);
    if (tid < kDv) fx.norm_w[tid] = nw;
    const float a_h = expf(a_log);
    __syncthreads();   // the mbarrier is initialised before anyone waits on it
    if (slot < 0 || slot >= p.num_slots) {
        // the same for every CTA of the cluster: all leave here
        if (tid == 0) {
            if (rank == 0) atomicOr(p.err_word, KDA_DEVERR_SLOT);
            mbar_wait_bounded(&fx.in_bar, 0, kWaitLimitNs);
        }
        cluster_wait();
        return;
    }
    ST *tile = reinterpret_cast<ST *>(p.state) + ((size_t)slot * H + h) * (kDk * kDv);
    float sv[16];
#pragma unroll
    for (int e = 0; e < 16; e++) sv[e] = (float)__ldcs(tile + (size_t)cluster_row<ST>(warp, e) * kDv + col);
    ConvItem cv[2];
#pragma unroll
    for (int it = 0; it < 2; it++) {
        if (it < n_items) {
            cv[it].tensor = it == 0 ? (tid < kDk ? 0 : 1) : 2;
            cv[it].ch = h * kDk + (tid & (kDk - 1));
#pragma unroll
            for (int j = 0; j < kTaps; j++)
                cv[it].win[j] = p.conv_state[(((size_t)slot * 3 + cv[it].tensor) * kTaps + j) * HC + cv[it].ch];
        }
    }
    const __nv_bfloat16 braw = tid == 224 ? p.beta[(size_t)b * H + h] : __nv_bfloat16();

    // ---- 3. gates (a wait that gives up is flagged; the CTA still takes part in the cluster
    //      barriers below and stores nothing)
    bool ok = true;
    {
        const bool arrived = mbar_wait_bounded(&fx.in_bar, 0, kWaitLimitNs);
        if (__syncthreads_or(!arrived)) {
            ok = false;
            if (tid == 0) {
                atomicOr(p.err_word, KDA_DEVERR_TIMEOUT);
                mbar_wait_bounded(&fx.in_bar, 0, kWaitLimitNs);
            }
        }
    }
    // a1: half-warp hw owns W rows 8 hw + j; lane li owns f_a entries [8 li, 8 li + 8)
    {
        const int b3 = (li >> 3) & 1, b2 = (li >> 2) & 1, b1 = (li >> 1) & 1;
        float f[8];
        unpack8(*reinterpret_cast<const uint4 *>(&fx.xs[4][li * 8]), f);
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const float *w = wreg[j];
            float a = w[0] * f[0];
#pragma unroll
            for (int e = 1; e < 8; e++) a = fmaf(w[e], f[e], a);
            acc[j] = a;
        }
        float v4[4], v2[2];
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const float keep = b3 ? acc[j + 4] : acc[j], give = b3 ? acc[j] : acc[j + 4];
            v4[j] = keep + __shfl_xor_sync(0xffffffffu, give, 8);
        }
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const float keep = b2 ? v4[j + 2] : v4[j], give = b2 ? v4[j] : v4[j + 2];
            v2[j] = keep + __shfl_xor_sync(0xffffffffu, give, 4);
        }
        float v1 = (b1 ? v2[1] : v2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? v2[0] : v2[1], 2);
        v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
        const int row = hw * 8 + 4 * b3 + 2 * b2 + b1;
        if ((li & 1) == 0) fx.alpha[row] = row_scaled<W8>(p, h, row, v1);
    }
    // a4: conv + SiLU, window shift
#pragma unroll
    for (int it = 0; it < 2; it++) {
        if (it < n_items) {
            const int tens = cv[it].tensor, c = cv[it].ch - h * kDk;
            float *dst = tens == 0 ? fx.q : (tens == 1 ? fx.k : fx.v);
            const __nv_bfloat16 x = fx.xs[tens][c];
            float acc = bf16_lo(cwr[it].x) * bf2f(cv[it].win[0]);
            acc = fmaf(bf16_hi(cwr[it].x), bf2f(cv[it].win[1]), acc);
            acc = fmaf(bf16_lo(cwr[it].y), bf2f(cv[it].win[2]), acc);
            acc = fmaf(bf16_hi(cwr[it].y), bf2f(x), acc);
            dst[c] = acc / (1.0f + expf(-acc));
            cv[it].win[0] = cv[it].win[1];
            cv[it].win[1] = cv[it].win[2];
            cv[it].win[2] = x;
        }
    }
    __syncthreads();
    // a2 decay, a5 norms and q.k, a3 beta
    if (tid < kDk) fx.alpha[tid] = expf(-a_h * softplusf_(fx.alpha[tid] + fx.dtb[tid]));
    if (warp >= 4 && warp < 7) {
        const int kind = warp - 4;
        const float *a = kind == 1 ? fx.k : fx.q;
        const float *c = kind == 0 ? fx.q : fx.k;
        const float4 x = *reinterpret_cast<const float4 *>(a + lane * 4);
        const float4 y = *reinterpret_cast<const float4 *>(c + lane * 4);
        float sum = x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
        sum = group_sum<32>(sum);
        if (lane == 0) fx.nrm[kind] = sum;
    }
    if (tid == 224) fx.nrm[3] = sigmoidf_(bf2f(braw));
    __syncthreads();

    // ---- 4. the sweep over this thread's 16 elements (decay, S^T k, S^T q)
    const float rq = rsqrtf((float)kDk) / sqrtf(fx.nrm[0] + p.l2_eps);
    const float rk = 1.0f / sqrtf(fx.nrm[1] + p.l2_eps);
    const float kq = fx.nrm[2] * rq * rk;
    const float beta = fx.nrm[3];
    float ak = 0.f, aq = 0.f;
    if constexpr (sizeof(ST) == 4) {
#pragma unroll
        for (int e = 0; e < 16; e++) {
            const int i = cluster_row<ST>(warp, e);
            const float a = fx.alpha[i], akk = a * (fx.k[i] * rk), aqq = a * (fx.q[i] * rq);
            ak = fmaf(sv[e], akk, ak);
            aq = fmaf(sv[e], aqq, aq);
            sv[e] *= a;
        }
    } else {
        float ak2 = 0.f, aq2 = 0.f;
#pragma unroll
        for (int e = 0; e < 16; e++) {
            const int i = cluster_row<ST>(warp, e);
            const float a = fx.alpha[i], akk = a * (fx.k[i] * rk), aqq = a * (fx.q[i] * rq);
            if (e < 8) {
                ak = fmaf(sv[e], akk, ak);
                aq = fmaf(sv[e], aqq, aq);
            } else {
                ak2 = fmaf(sv[e], akk, ak2);
                aq2 = fmaf(sv[e], aqq, aq2);
            }
            sv[e] *= a;
        }
        ak += ak2;
        aq += aq2;
    }
    fx.red[warp][0][lane] = ak;
    fx.red[warp][1][lane] = aq;
    __syncthreads();
    cluster_wait();   // every CTA of the cluster has started
    float o = 0.f;
    if (warp == 0) {
        float stk = 0.f, stq = 0.f;
#pragma unroll
        for (int w = 0; w < NT / 32; w++) { stk += fx.red[w][0][lane]; stq += fx.red[w][1][lane]; }
        const float u = fx.v[col] - stk;
        o = stq + beta * u * kq;
        fx.u[lane] = u;
    }
    __syncthreads();   // fx.u is written
    // ---- 5. the RMS norm needs the sum of o^2 over the 128 columns.  Rank c's 32 columns are
    //      summed here exactly as warp c of the one-tile kernel sums them, and that one value
    //      goes into every CTA of the cluster; while it travels, every warp writes its part of
    //      S += beta k u^T back to the slot (rounded once to the storage dtype) and rank 0 the
    //      conv window.  A CTA whose inputs never arrived (ok false) stores nothing but still
    //      takes part in the cluster barrier.
    if (warp == 0) {
        const float ss = group_sum<32>(o * o);
        if (lane < kClusterN) st_cluster_f32(map_to_rank(&fx.rms[rank], (uint32_t)lane), ss);
    }
    cluster_arrive();
    if (ok) {
        const float uu = fx.u[lane];
#pragma unroll
        for (int e = 0; e < 16; e++) {
            const int i = cluster_row<ST>(warp, e);
            const float bk = beta * fx.k[i] * rk;
            const float nv = fmaf(bk, uu, sv[e]);
            if constexpr (sizeof(ST) == 4) __stcs(tile + (size_t)i * kDv + col, nv);
            else tile[(size_t)i * kDv + col] = __float2bfloat16_rn(nv);
        }
        if (rank == 0) {
#pragma unroll
            for (int it = 0; it < 2; it++) {
                if (it < n_items) {
#pragma unroll
                    for (int j = 0; j < kTaps; j++)
                        p.conv_state[(((size_t)slot * 3 + cv[it].tensor) * kTaps + j) * HC + cv[it].ch] = cv[it].win[j];
                }
            }
        }
    }
    cluster_wait();   // fx.rms holds the four partial sums
    if (ok && warp == 0) {
        const float ms = (fx.rms[0] + fx.rms[1] + fx.rms[2] + fx.rms[3]) * (1.0f / kDv);
        const float y = o * rsqrtf(ms + p.norm_eps) * fx.norm_w[col] * sigmoidf_(bf2f(fx.xs[3][col]));
        p.out[(size_t)b * (H * kDv) + (size_t)h * kDv + col] = __float2bfloat16_rn(y);
    }
}

// SMs of the current device (cached per device).
cudaError_t device_sms(int *sms)
{
    static std::atomic<int> cache[KernelSetup::kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= KernelSetup::kMaxDevices) return cudaErrorInvalidDevice;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    *sms = n;
    return cudaSuccess;
}

template <typename ST, bool W8>
cudaError_t launch_decode_cluster(const RecurrentParams &p, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.H * kClusterN), (unsigned)p.B);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = kClusterN;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kda_decode_cluster_kernel<ST, W8>, p);
}

template <bool W8, bool RESUME>
cudaError_t launch_decode_pair_t(const RecurrentParams &p_in, cudaStream_t stream)
{
    static KernelSetup setup;
    cudaError_t e = setup.get(kda_decode_pair_kernel<W8, RESUME>, NT, pair_smem(), 0, nullptr);
    if (e != cudaSuccess) return e;
    RecurrentParams p = p_in;
    p.prefetch_stride = 0;
    p.prefetch_early = 0;
    return launch_pdl(kda_decode_pair_kernel<W8, RESUME>, dim3((unsigned)p.H, (unsigned)((p.B + 1) / 2)), dim3(NT),
                      pair_smem(), stream, p);
}

template <bool W8>
cudaError_t launch_decode_pair(const RecurrentParams &p, cudaStream_t stream)
{
    return p.prev_accepted ? launch_decode_pair_t<W8, true>(p, stream) : launch_decode_pair_t<W8, false>(p, stream);
}

template <typename ST, bool W8>
cudaError_t launch_decode_t(const RecurrentParams &p_in, cudaStream_t stream)
{
    static KernelSetup setup;
    const size_t smem = decode_smem<ST>();
    int resident = 0;
    cudaError_t e = setup.get(kda_decode_kernel<ST, W8>, NT, smem, 0, &resident);
    if (e != cudaSuccess) return e;
    RecurrentParams p = p_in;
    p.prefetch_stride = resident;   // the next-wave prefetch is issued after the gates
    return launch_pdl(kda_decode_kernel<ST, W8>, dim3((unsigned)p.H, (unsigned)p.B), dim3(NT), smem, stream, p);
}

// CTAs of the tile kernel (for G staged tokens) that the current device holds at once.
template <typename ST, bool RECORDS, bool W8>
cudaError_t tile_setup(int G, size_t smem, int *resident)
{
    static KernelSetup setup;
    return setup.get(kda_tile_kernel<ST, RECORDS, W8>, NT, smem, G, resident);
}

template <typename ST, bool RECORDS, bool W8>
cudaError_t launch_t(const RecurrentParams &p_in, cudaStream_t stream)
{
    const int G = p_in.T < kGroup ? p_in.T : kGroup;
    const size_t smem = smem_total(G);
    int resident = 0;   // CTAs of this kernel the GPU holds at once
    cudaError_t e = tile_setup<ST, RECORDS, W8>(G, smem, &resident);
    if (e != cudaSuccess) return e;
    RecurrentParams p = p_in;
    p.prefetch_stride = resident;
    // many waves: prefetch at CTA start; one or two: after the gates (measured on GB300)
    p.prefetch_early = (long)p.B * p.H >= 3L * resident ? 1 : 0;
    return launch_pdl(kda_tile_kernel<ST, RECORDS, W8>, dim3((unsigned)p.H, (unsigned)p.B), dim3(NT), smem, stream, p);
}

template <bool W8>
cudaError_t dispatch_recurrent(const RecurrentParams &p, bool bf16_state, bool records, cudaStream_t stream)
{
    // Single-token decode.  BF16 tiles: the 4-CTA/SM decode kernel (measured on GB300, 256 x 32
    // tiles: 110 us per launch, against 174 us on the tile kernel).  FP32 tiles: the register-
    // resident tile kernel while one resident wave of it holds every tile, two tiles per CTA
    // beyond that (64 x 8 tiles: 14.1 us per launch in steady state and 20.0 us cold with tile
    // pairs, against 16.6 and 23.3 us with one tile per CTA; the 4-CTA/SM layout measured 18.1
    // us steady and is not used for FP32).
    // Few tiles (each cluster of four CTAs per tile still fits on the SMs): one tile per
    // cluster, the columns split over its CTAs.
    if (!records && p.T == 1 && !p.prev_accepted && !p.n_tokens) {
        int sms = 0;
        const cudaError_t e = device_sms(&sms);
        if (e != cudaSuccess) return e;
        if ((long)p.B * p.H * kClusterN <= sms)
            return bf16_state ? launch_decode_cluster<__nv_bfloat16, W8>(p, stream) : launch_decode_cluster<float, W8>(p, stream);
    }
    if (!records && p.T == 1 && bf16_state && !p.prev_accepted) return launch_decode_t<__nv_bfloat16, W8>(p, stream);
    if (!records && p.T == 1 && !bf16_state && !p.n_tokens) {   // decode, or decode resuming from records
        int tile_resident = 0;
        const cudaError_t e = tile_setup<float, false, W8>(1, smem_total(1), &tile_resident);
        if (e != cudaSuccess) return e;
        if ((long)p.B * p.H > tile_resident) return launch_decode_pair<W8>(p, stream);
    }
    if (bf16_state) return records ? launch_t<__nv_bfloat16, true, W8>(p, stream) : launch_t<__nv_bfloat16, false, W8>(p, stream);
    return records ? launch_t<float, true, W8>(p, stream) : launch_t<float, false, W8>(p, stream);
}

}  // namespace

cudaError_t launch_recurrent(const RecurrentParams &p, bool bf16_state, bool records, cudaStream_t stream)
{
    // FP8 E4M3 W_fb (per-row scales) runs its own instances of the same kernels
    return p.W_fb8 ? dispatch_recurrent<true>(p, bf16_state, records, stream)
                   : dispatch_recurrent<false>(p, bf16_state, records, stream);
}

}  // namespace kda
