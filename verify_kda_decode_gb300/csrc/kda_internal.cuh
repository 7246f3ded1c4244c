// kda_internal.cuh -- declarations shared by the libkda translation units (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/kda.h"

namespace kda {

constexpr int kDk = 128;       // key head dim
constexpr int kDv = 128;       // value head dim
constexpr int kRank = 128;     // f_a rank
constexpr int kConv = 4;       // conv taps
constexpr int kTaps = kConv - 1;
constexpr int kMaxVerifyT = 16;

// Everything a recurrent (token-serial) launch needs.  Token (b, t) of an input with C
// channels per token lives at ((b * T + t) * C); decode is the T = 1 case.
struct RecurrentParams {
    // layer
    int H;
    const __nv_bfloat16 *W_fb;      // [H*128, 128] BF16 weights, or null with FP8 weights
    const uint8_t *W_fb8;           // [H*128, 128] FP8 E4M3 codes, or null with BF16 weights
    const float *W_fb_scale;        // [H*128] per-row scales of the FP8 codes
    const float *A_log;             // [H]
    const float *dt_bias;           // [H*128]
    const __nv_bfloat16 *conv_w;    // [3, H*128, 4]
    const float *norm_w;            // [128]
    float l2_eps, norm_eps;
    // pool
    void *state;                    // [num_slots, H, 128, 128]
    __nv_bfloat16 *conv_state;      // [num_slots, 3, 3, H*128]
    int num_slots;
    int *err_word;
    // call
    const int *slot_ids;            // [B]
    int B, T;
    const __nv_bfloat16 *q, *k, *v, *f_a, *beta, *gate;
    __nv_bfloat16 *out;             // [B, T, H*128]
    float *rec_state;               // verify: [B, T, H, 128, 128]
    __nv_bfloat16 *rec_conv;        // verify: [B, T, 3, 3, H*128]
    // resume (optional): start sequence b from record prev_accepted[b] - 1 of the previous
    // step's records instead of its slot; with records on, that record is also committed
    const int *prev_accepted;       // [B] or null
    int prev_T;
    const float *prev_rec_state;    // [B, prev_T, H, 128, 128]
    const __nv_bfloat16 *prev_rec_conv;   // [B, prev_T, 3, 3, H*128]
    const int *n_tokens;            // [B] tokens of sequence b (1..T), or null for T
    // variable-length prefill (optional): sequence b is tokens [cu_seqlens[b], cu_seqlens[b+1])
    // of packed inputs with total_tokens rows, T then bounds every length; null: sequence b is
    // tokens [b*T, (b+1)*T)
    const int *cu_seqlens;
    int total_tokens;
    int prefetch_stride;            // CTAs resident at once (set by the launcher; 0 = none)
    int prefetch_early;             // 1: prefetch the next wave's tile at CTA start
};

// 8 FP8 E4M3 codes (byte e = element e) -> 8 floats.  Exact: every E4M3 value is a half.
__device__ __forceinline__ void e4m3x8_to_f32(uint2 c, float *f)
{
    const uint32_t w[2] = {c.x, c.y};
#pragma unroll
    for (int i = 0; i < 2; i++) {
#pragma unroll
        for (int hf = 0; hf < 2; hf++) {
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)((w[i] >> (16 * hf)) & 0xffffu), __NV_E4M3);
            const float2 v = __half22float2(__half2(hr));
            f[4 * i + 2 * hf] = v.x;
            f[4 * i + 2 * hf + 1] = v.y;
        }
    }
}

// Launchers (kda_tile.cu, kda_commit.cu).  `records` selects verify semantics (records
// written, pool untouched unless resuming); otherwise the final state and window are written
// back to the slot (decode).
cudaError_t launch_recurrent(const RecurrentParams &p, bool bf16_state, bool records,
                             cudaStream_t stream);

struct CommitParams {
    void *state;                    // [num_slots, H, 128, 128]
    __nv_bfloat16 *conv_state;      // [num_slots, 3, 3, H*128]
    int num_slots, H;
    int *err_word;
    const int *slot_ids, *accepted;
    int B, T;
    const float *rec_state;         // [B, T, H, 128, 128]
    const __nv_bfloat16 *rec_conv;  // [B, T, 3, 3, H*128]
};

cudaError_t launch_commit(const CommitParams &p, bool bf16_state, cudaStream_t stream);

// Per-device launch set-up of one kernel.  A function's dynamic shared-memory limit belongs to
// a device's context, and how many CTAs of the kernel a device holds at once depends on its SM
// count, so both are kept per device ordinal (the current device at launch time), for up to
// kSlots shared-memory variants of the kernel.  Thread-safe: the common path is one atomic load.
class KernelSetup {
  public:
    static constexpr int kMaxDevices = 64;
    static constexpr int kSlots = 17;

    // Raises the kernel's shared-memory limit to `smem` on the current device (once) and
    // returns in *resident the CTAs of `threads` threads and `smem` bytes the device holds.
    template <typename Kern>
    cudaError_t get(Kern kern, int threads, size_t smem, int slot, int *resident)
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= kMaxDevices || slot < 0 || slot >= kSlots) return cudaErrorInvalidValue;
        int r = resident_[dev][slot].load(std::memory_order_acquire);
        if (r == 0) {
            std::lock_guard<std::mutex> lock(mu_);
            r = resident_[dev][slot].load(std::memory_order_relaxed);
            if (r == 0) {
                if (smem_[dev].load(std::memory_order_relaxed) < (long)smem) {
                    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
                    if (e != cudaSuccess) return e;
                    smem_[dev].store((long)smem, std::memory_order_relaxed);
                }
                int sms = 0, per_sm = 0;
                e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
                if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
                if (e != cudaSuccess) return e;
                r = sms * per_sm + 1;
                resident_[dev][slot].store(r, std::memory_order_release);
            }
        }
        if (resident) *resident = r - 1;
        return cudaSuccess;
    }

  private:
    std::atomic<long> smem_[kMaxDevices];
    std::atomic<int> resident_[kMaxDevices][kSlots];   // resident CTAs + 1; 0 = not set up
    std::mutex mu_;
};

// Launches `kern` with programmatic stream serialization: it may start while the previous
// kernel on the stream drains.  Kernels launched this way read layer weights (which no kernel
// writes) before grid_dependency_wait() and everything else, for use, after it; the one read
// before it of data a previous kernel may write (a slot id or accepted length) only picks the
// address of an L2 prefetch, and the value used is read again after the wait.
template <typename Kern, typename Arg>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, const Arg &arg)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, arg);
}

}  // namespace kda
