// kda_prefill.cu -- prefill over whole prompts.
//
// First form: the token-serial recurrence over all L tokens in one launch (the decode kernel's
// loop with T = L), state kept in FP32 registers throughout and written back once.
#include "kda_prefill.cuh"

namespace kda {

size_t prefill_workspace_bytes(int, int, int) { return 0; }

cudaError_t launch_prefill(const RecurrentParams &p, bool bf16_state, void *, cudaStream_t stream)
{
    return launch_recurrent(p, bf16_state, false, stream);
}

}  // namespace kda
