// kda_prefill.cuh -- prefill launcher interface (internal).
#pragma once

#include "kda_internal.cuh"

namespace kda {

constexpr int kPrefillChunk = 64;   // tokens per chunk of the chunked form

// Scratch bytes a prefill of B sequences x L tokens needs (0 when none).
size_t prefill_workspace_bytes(int H, int B, int L);

// Scratch bytes of a variable-length prefill of B sequences with total_tokens tokens in all.
size_t prefill_varlen_workspace_bytes(int H, int B, long total_tokens);

// Prefill from the slots' state and window: p.T = L, or, with p.cu_seqlens, the longest
// sequence's length bound.  `workspace` holds at least the matching *_workspace_bytes.
cudaError_t launch_prefill(const RecurrentParams &p, bool bf16_state, void *workspace,
                           cudaStream_t stream);

}  // namespace kda
