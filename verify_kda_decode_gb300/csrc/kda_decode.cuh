// kda_decode.cuh -- persistent decode / verify launcher (internal).
#pragma once

#include "kda_internal.cuh"

namespace kda {

// Decode (records = false: state and window written back to the slot) or verify (records =
// true: FP32 state and window recorded after each of the p.T tokens, slot untouched) with the
// persistent, bulk-copy-pipelined kernel.  1 <= p.T <= kMaxVerifyT.
cudaError_t launch_stream(const RecurrentParams &p, bool bf16_state, bool records, cudaStream_t stream);

// Dynamic shared memory the kernel uses for a given T.
size_t stream_smem_bytes(bool bf16_state, int T);

}  // namespace kda
