// kda_prefill.cuh -- prefill launcher interface (internal).
#pragma once

#include "kda_internal.cuh"

namespace kda {

constexpr int kPrefillChunk = 64;   // tokens per chunk of the chunked form

// Scratch bytes a prefill of B sequences x L tokens needs (0 when none).
size_t prefill_workspace_bytes(int H, int B, int L);

// Prefill from the slots' state and window; p.T = L.  `workspace` holds at least
// prefill_workspace_bytes(p.H, p.B, p.T) bytes.
cudaError_t launch_prefill(const RecurrentParams &p, bool bf16_state, void *workspace,
                           cudaStream_t stream);

}  // namespace kda
