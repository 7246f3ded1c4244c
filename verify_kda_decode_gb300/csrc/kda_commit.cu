// kda_commit.cu -- commit of accepted draft lengths after a verify launch.
//
// For sequence b with n = accepted[b] >= 1 the slot takes the FP32 record written after draft
// token n-1 (a bit copy into an FP32 pool, round-to-nearest-even into a BF16 pool: "typed state
// stores", NVFP4 Kimi K3 targets page, Description) and the conv window recorded after that
// token.  n = 0 leaves the slot as it was.  One CTA per (sequence, head) moves the 64 KiB FP32
// record tile with 128-bit loads and stores, and the conv-window rows with loads issued beside
// the tile's (measured on GB300, verify_b64's drawn lengths: 14.4 -> 12.3 us per launch against
// copying the window after the tile); pure data movement, bound by HBM.
#include "kda_internal.cuh"
#include "kda_ptx.cuh"

namespace kda {
namespace {

constexpr int NT = 256;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

template <bool BF16>
__global__ void __launch_bounds__(NT, 3) kda_commit_kernel(const CommitParams p)
{
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, H = p.H, HC = H * kDk;
    grid_dependency_wait();   // the records come from the verify launch before this one
    const int n = p.accepted[b], slot = p.slot_ids[b];
    if (n < 0 || n > p.T) {
        if (tid == 0 && h == 0) atomicOr(p.err_word, KDA_DEVERR_ACCEPTED);
        return;
    }
    if (slot < 0 || slot >= p.num_slots) {
        if (tid == 0 && h == 0) atomicOr(p.err_word, KDA_DEVERR_SLOT);
        return;
    }
    if (n == 0) return;
    const size_t rec_tok = (size_t)b * p.T + (n - 1);
    const float4 *src = reinterpret_cast<const float4 *>(p.rec_state + (rec_tok * H + h) * (size_t)(kDk * kDv));
    constexpr int N4 = kDk * kDv / 4;   // float4 per tile
    static_assert(N4 % NT == 0, "tile split");
    // every thread issues all 16 of its 128-bit loads before the first store
    constexpr int PER = N4 / NT;   // 16
    float4 v[PER];
#pragma unroll
    for (int j = 0; j < PER; j++) v[j] = __ldcs(src + tid + j * NT);
    // this head's channels of the conv window (3 tensors x 3 taps x 128 channels), loaded with
    // the tile so that their round trip overlaps it
    // (thread tid takes rows tid / 128 + 2 q of the 9, channel tid % 128)
    static_assert(NT == 2 * kDk, "two window rows per pass");
    constexpr int NW = (3 * kTaps + 1) / 2;   // 5 passes, the last on half the threads
    const int wr0 = tid / kDk, wc = tid % kDk;
    const __nv_bfloat16 *wsrc = p.rec_conv + (rec_tok * 3 * kTaps + wr0) * HC + h * kDk + wc;
    __nv_bfloat16 w[NW];
#pragma unroll
    for (int q = 0; q < NW; q++)
        if (wr0 + 2 * q < 3 * kTaps) w[q] = wsrc[(size_t)2 * q * HC];
    if (!BF16) {
        float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.state) + ((size_t)slot * H + h) * (kDk * kDv));
#pragma unroll
        for (int j = 0; j < PER; j++) __stcs(dst + tid + j * NT, v[j]);
    } else {
        // float4 j of the tile holds elements 4 (tid + j NT) .. +3: store them as 4 bf16 (8 bytes)
        uint2 *dst = reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.state) + ((size_t)slot * H + h) * (kDk * kDv));
#pragma unroll
        for (int j = 0; j < PER; j++)
            __stcs(dst + tid + j * NT, make_uint2(pack_bf16x2(v[j].x, v[j].y), pack_bf16x2(v[j].z, v[j].w)));
    }
    __nv_bfloat16 *wdst = p.conv_state + ((size_t)slot * 3 * kTaps + wr0) * HC + h * kDk + wc;
#pragma unroll
    for (int q = 0; q < NW; q++)
        if (wr0 + 2 * q < 3 * kTaps) wdst[(size_t)2 * q * HC] = w[q];
}

}  // namespace

cudaError_t launch_commit(const CommitParams &p, bool bf16_state, cudaStream_t stream)
{
    const dim3 grid((unsigned)p.H, (unsigned)p.B), block(NT);
    return bf16_state ? launch_pdl(kda_commit_kernel<true>, grid, block, 0, stream, p)
                      : launch_pdl(kda_commit_kernel<false>, grid, block, 0, stream, p);
}

}  // namespace kda
