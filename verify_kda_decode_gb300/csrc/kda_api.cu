// kda_api.cu -- the extern "C" entry points of libkda: argument checks, then kernel launches.
// No entry point allocates memory, synchronises (except kda_get_error) or reads device memory
// on the host, so calls can be captured in CUDA graphs ("stateful entries take caller-owned
// state created before capture", Kimi K3 on modeling_v2 page, section 1).
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "kda_internal.cuh"
#include "kda_prefill.cuh"

namespace {

thread_local char g_msg[256] = "";

kda_status fail(kda_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return s;
}

bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define REQUIRE_PTR(p)                                                                    \
    do {                                                                                  \
        if (!aligned16(p)) return fail(KDA_ERR_INVALID_ARG, "%s is null or not 16-byte aligned", #p); \
    } while (0)

kda_status check_layer(const kda_layer *L)
{
    if (!L) return fail(KDA_ERR_INVALID_ARG, "layer is null");
    if (L->num_heads < 1 || L->num_heads > 4096)
        return fail(KDA_ERR_INVALID_ARG, "num_heads=%d outside [1, 4096]", L->num_heads);
    if (L->head_k_dim != kda::kDk || L->head_v_dim != kda::kDv || L->fa_rank != kda::kRank ||
        L->conv_size != kda::kConv)
        return fail(KDA_ERR_UNSUPPORTED, "only dk=dv=128, r=128, conv_size=4 are built (got %d,%d,%d,%d)",
                    L->head_k_dim, L->head_v_dim, L->fa_rank, L->conv_size);
    REQUIRE_PTR(L->W_fb);
    if (L->w_fb_dtype != KDA_W_BF16 && L->w_fb_dtype != KDA_W_FP8_E4M3)
        return fail(KDA_ERR_INVALID_ARG, "w_fb_dtype=%d is neither KDA_W_BF16 nor KDA_W_FP8_E4M3", L->w_fb_dtype);
    if (L->w_fb_dtype == KDA_W_FP8_E4M3) REQUIRE_PTR(L->W_fb_scale);
    REQUIRE_PTR(L->A_log);
    REQUIRE_PTR(L->dt_bias);
    REQUIRE_PTR(L->conv_w);
    REQUIRE_PTR(L->norm_w);
    if (!(L->l2_eps >= 0.f) || !(L->norm_eps >= 0.f))
        return fail(KDA_ERR_INVALID_ARG, "epsilons must be >= 0");
    return KDA_OK;
}

kda_status check_pool(const kda_pool *P)
{
    if (!P) return fail(KDA_ERR_INVALID_ARG, "pool is null");
    REQUIRE_PTR(P->state);
    REQUIRE_PTR(P->conv_state);
    if (!P->err_word || (reinterpret_cast<uintptr_t>(P->err_word) & 3u))
        return fail(KDA_ERR_INVALID_ARG, "err_word is null or misaligned");
    if (P->state_dtype != KDA_STATE_F32 && P->state_dtype != KDA_STATE_BF16)
        return fail(KDA_ERR_INVALID_ARG, "state_dtype=%d is neither KDA_STATE_F32 nor KDA_STATE_BF16", P->state_dtype);
    if (P->num_slots < 1) return fail(KDA_ERR_INVALID_ARG, "num_slots=%d < 1", P->num_slots);
    return KDA_OK;
}

kda_status check_batch(const kda_pool *P, int32_t B)
{
    if (B < 0) return fail(KDA_ERR_INVALID_ARG, "B=%d < 0", B);
    if (B > P->num_slots) return fail(KDA_ERR_INVALID_ARG, "B=%d exceeds num_slots=%d (slots must be distinct)", B, P->num_slots);
    if (B > 65535) return fail(KDA_ERR_UNSUPPORTED, "B=%d > 65535", B);
    return KDA_OK;
}

kda_status launched(cudaError_t e)
{
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "CUDA: %s", cudaGetErrorString(e));
    g_msg[0] = '\0';
    return KDA_OK;
}

kda::RecurrentParams recurrent_params(const kda_layer *L, const kda_pool *P, const int32_t *slot_ids,
                                      int32_t B, int32_t T, const void *q, const void *k,
                                      const void *v, const void *f_a, const void *beta,
                                      const void *gate, void *out)
{
    kda::RecurrentParams p;
    memset(&p, 0, sizeof p);
    p.H = L->num_heads;
    const bool fp8 = L->w_fb_dtype == KDA_W_FP8_E4M3;
    p.W_fb = fp8 ? nullptr : static_cast<const __nv_bfloat16 *>(L->W_fb);
    p.W_fb8 = fp8 ? static_cast<const uint8_t *>(L->W_fb) : nullptr;
    p.W_fb_scale = fp8 ? L->W_fb_scale : nullptr;
    p.A_log = L->A_log;
    p.dt_bias = L->dt_bias;
    p.conv_w = static_cast<const __nv_bfloat16 *>(L->conv_w);
    p.norm_w = L->norm_w;
    p.l2_eps = L->l2_eps;
    p.norm_eps = L->norm_eps;
    p.state = P->state;
    p.conv_state = static_cast<__nv_bfloat16 *>(P->conv_state);
    p.num_slots = P->num_slots;
    p.err_word = P->err_word;
    p.slot_ids = slot_ids;
    p.B = B;
    p.T = T;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = static_cast<const __nv_bfloat16 *>(k);
    p.v = static_cast<const __nv_bfloat16 *>(v);
    p.f_a = static_cast<const __nv_bfloat16 *>(f_a);
    p.beta = static_cast<const __nv_bfloat16 *>(beta);
    p.gate = static_cast<const __nv_bfloat16 *>(gate);
    p.out = static_cast<__nv_bfloat16 *>(out);
    return p;
}

#define CHECK(expr)                          \
    do {                                     \
        kda_status s_ = (expr);              \
        if (s_ != KDA_OK) return s_;         \
    } while (0)

kda_status check_token_inputs(const void *slot_ids, const void *q, const void *k, const void *v,
                              const void *f_a, const void *beta, const void *gate, const void *out)
{
    if (!slot_ids || (reinterpret_cast<uintptr_t>(slot_ids) & 3u))
        return fail(KDA_ERR_INVALID_ARG, "slot_ids is null or misaligned");
    REQUIRE_PTR(q);
    REQUIRE_PTR(k);
    REQUIRE_PTR(v);
    REQUIRE_PTR(f_a);
    if (!beta || (reinterpret_cast<uintptr_t>(beta) & 1u)) return fail(KDA_ERR_INVALID_ARG, "beta_logit is null or misaligned");
    REQUIRE_PTR(gate);
    REQUIRE_PTR(out);
    return KDA_OK;
}

// The previous step's records of a resume call: all absent, or accepted lengths plus records.
kda_status check_prev(const int32_t *prev_accepted, int32_t prev_T, const float *prev_rec_state,
                      const void *prev_rec_conv)
{
    if (!prev_accepted) return KDA_OK;
    if (reinterpret_cast<uintptr_t>(prev_accepted) & 3u) return fail(KDA_ERR_INVALID_ARG, "prev_accepted is misaligned");
    if (prev_T < 1 || prev_T > kda::kMaxVerifyT)
        return fail(KDA_ERR_INVALID_ARG, "prev_T=%d outside [1, %d]", prev_T, kda::kMaxVerifyT);
    REQUIRE_PTR(prev_rec_state);
    REQUIRE_PTR(prev_rec_conv);
    return KDA_OK;
}

void set_prev(kda::RecurrentParams &p, const int32_t *prev_accepted, int32_t prev_T,
              const float *prev_rec_state, const void *prev_rec_conv)
{
    if (!prev_accepted) return;
    p.prev_accepted = prev_accepted;
    p.prev_T = prev_T;
    p.prev_rec_state = prev_rec_state;
    p.prev_rec_conv = static_cast<const __nv_bfloat16 *>(prev_rec_conv);
}

}  // namespace

// Lets other translation units of the library report a host-side argument error through
// kda_last_error().
void kda_set_last_error(const char *msg)
{
    snprintf(g_msg, sizeof g_msg, "%s", msg);
}

extern "C" {

kda_status kda_decode(const kda_layer *layer, const kda_pool *pool, const int32_t *slot_ids,
                      int32_t B, const void *q, const void *k, const void *v, const void *f_a,
                      const void *beta_logit, const void *gate, void *out, void *stream)
{
    CHECK(check_layer(layer));
    CHECK(check_pool(pool));
    CHECK(check_batch(pool, B));
    if (B == 0) return launched(cudaSuccess);
    CHECK(check_token_inputs(slot_ids, q, k, v, f_a, beta_logit, gate, out));
    const kda::RecurrentParams p = recurrent_params(layer, pool, slot_ids, B, 1, q, k, v, f_a, beta_logit, gate, out);
    return launched(kda::launch_recurrent(p, pool->state_dtype == KDA_STATE_BF16, false,
                                          static_cast<cudaStream_t>(stream)));
}

kda_status kda_verify(const kda_layer *layer, const kda_pool *pool, const int32_t *slot_ids,
                      int32_t B, int32_t T, const void *q, const void *k, const void *v,
                      const void *f_a, const void *beta_logit, const void *gate, void *out,
                      float *rec_state, void *rec_conv, void *stream)
{
    CHECK(check_layer(layer));
    CHECK(check_pool(pool));
    CHECK(check_batch(pool, B));
    if (T < 1 || T > kda::kMaxVerifyT) return fail(KDA_ERR_INVALID_ARG, "T=%d outside [1, %d]", T, kda::kMaxVerifyT);
    if (B == 0) return launched(cudaSuccess);
    CHECK(check_token_inputs(slot_ids, q, k, v, f_a, beta_logit, gate, out));
    REQUIRE_PTR(rec_state);
    REQUIRE_PTR(rec_conv);
    kda::RecurrentParams p = recurrent_params(layer, pool, slot_ids, B, T, q, k, v, f_a, beta_logit, gate, out);
    p.rec_state = rec_state;
    p.rec_conv = static_cast<__nv_bfloat16 *>(rec_conv);
    return launched(kda::launch_recurrent(p, pool->state_dtype == KDA_STATE_BF16, true,
                                          static_cast<cudaStream_t>(stream)));
}

kda_status kda_decode_resume(const kda_layer *layer, const kda_pool *pool, const int32_t *slot_ids,
                             int32_t B, const int32_t *prev_accepted, int32_t prev_T,
                             const float *prev_rec_state, const void *prev_rec_conv,
                             const void *q, const void *k, const void *v, const void *f_a,
                             const void *beta_logit, const void *gate, void *out, void *stream)
{
    CHECK(check_layer(layer));
    CHECK(check_pool(pool));
    CHECK(check_batch(pool, B));
    CHECK(check_prev(prev_accepted, prev_T, prev_rec_state, prev_rec_conv));
    if (B == 0) return launched(cudaSuccess);
    CHECK(check_token_inputs(slot_ids, q, k, v, f_a, beta_logit, gate, out));
    kda::RecurrentParams p = recurrent_params(layer, pool, slot_ids, B, 1, q, k, v, f_a, beta_logit, gate, out);
    set_prev(p, prev_accepted, prev_T, prev_rec_state, prev_rec_conv);
    return launched(kda::launch_recurrent(p, pool->state_dtype == KDA_STATE_BF16, false,
                                          static_cast<cudaStream_t>(stream)));
}

kda_status kda_verify_resume(const kda_layer *layer, const kda_pool *pool, const int32_t *slot_ids,
                             int32_t B, int32_t T, const int32_t *n_tokens,
                             const int32_t *prev_accepted, int32_t prev_T,
                             const float *prev_rec_state, const void *prev_rec_conv,
                             const void *q, const void *k, const void *v, const void *f_a,
                             const void *beta_logit, const void *gate, void *out,
                             float *rec_state, void *rec_conv, void *stream)
{
    CHECK(check_layer(layer));
    CHECK(check_pool(pool));
    CHECK(check_batch(pool, B));
    if (T < 1 || T > kda::kMaxVerifyT) return fail(KDA_ERR_INVALID_ARG, "T=%d outside [1, %d]", T, kda::kMaxVerifyT);
    if (n_tokens && (reinterpret_cast<uintptr_t>(n_tokens) & 3u)) return fail(KDA_ERR_INVALID_ARG, "n_tokens is misaligned");
    CHECK(check_prev(prev_accepted, prev_T, prev_rec_state, prev_rec_conv));
    if (B == 0) return launched(cudaSuccess);
    CHECK(check_token_inputs(slot_ids, q, k, v, f_a, beta_logit, gate, out));
    REQUIRE_PTR(rec_state);
    REQUIRE_PTR(rec_conv);
    if (prev_accepted && (static_cast<const void *>(prev_rec_state) == static_cast<const void *>(rec_state) ||
                          prev_rec_conv == rec_conv))
        return fail(KDA_ERR_INVALID_ARG, "the previous records and this step's records must be different buffers");
    kda::RecurrentParams p = recurrent_params(layer, pool, slot_ids, B, T, q, k, v, f_a, beta_logit, gate, out);
    p.rec_state = rec_state;
    p.rec_conv = static_cast<__nv_bfloat16 *>(rec_conv);
    p.n_tokens = n_tokens;
    set_prev(p, prev_accepted, prev_T, prev_rec_state, prev_rec_conv);
    return launched(kda::launch_recurrent(p, pool->state_dtype == KDA_STATE_BF16, true,
                                          static_cast<cudaStream_t>(stream)));
}

kda_status kda_commit(const kda_pool *pool, int32_t num_heads, int32_t head_k_dim,
                      int32_t head_v_dim, int32_t conv_size, const int32_t *slot_ids,
                      const int32_t *accepted, int32_t B, int32_t T, const float *rec_state,
                      const void *rec_conv, void *stream)
{
    CHECK(check_pool(pool));
    if (num_heads < 1 || num_heads > 4096) return fail(KDA_ERR_INVALID_ARG, "num_heads=%d outside [1, 4096]", num_heads);
    if (head_k_dim != kda::kDk || head_v_dim != kda::kDv || conv_size != kda::kConv)
        return fail(KDA_ERR_UNSUPPORTED, "only dk=dv=128, conv_size=4 are built");
    CHECK(check_batch(pool, B));
    if (T < 1 || T > kda::kMaxVerifyT) return fail(KDA_ERR_INVALID_ARG, "T=%d outside [1, %d]", T, kda::kMaxVerifyT);
    if (B == 0) return launched(cudaSuccess);
    if (!slot_ids || (reinterpret_cast<uintptr_t>(slot_ids) & 3u)) return fail(KDA_ERR_INVALID_ARG, "slot_ids is null or misaligned");
    if (!accepted || (reinterpret_cast<uintptr_t>(accepted) & 3u)) return fail(KDA_ERR_INVALID_ARG, "accepted is null or misaligned");
    REQUIRE_PTR(rec_state);
    REQUIRE_PTR(rec_conv);
    kda::CommitParams p;
    p.state = pool->state;
    p.conv_state = static_cast<__nv_bfloat16 *>(pool->conv_state);
    p.num_slots = pool->num_slots;
    p.H = num_heads;
    p.err_word = pool->err_word;
    p.slot_ids = slot_ids;
    p.accepted = accepted;
    p.B = B;
    p.T = T;
    p.rec_state = rec_state;
    p.rec_conv = static_cast<const __nv_bfloat16 *>(rec_conv);
    return launched(kda::launch_commit(p, pool->state_dtype == KDA_STATE_BF16, static_cast<cudaStream_t>(stream)));
}

size_t kda_prefill_workspace_size(const kda_layer *layer, int32_t B, int32_t L, int32_t chunk)
{
    if (!layer || B < 0 || L < 0 || chunk != kda::kPrefillChunk) return 0;
    return kda::prefill_workspace_bytes(layer->num_heads, B, L);
}

kda_status kda_prefill(const kda_layer *layer, const kda_pool *pool, const int32_t *slot_ids,
                       int32_t B, int32_t L, int32_t chunk, const void *q, const void *k,
                       const void *v, const void *f_a, const void *beta_logit, const void *gate,
                       void *out, void *workspace, size_t workspace_bytes, void *stream)
{
    CHECK(check_layer(layer));
    CHECK(check_pool(pool));
    CHECK(check_batch(pool, B));
    if (chunk != kda::kPrefillChunk) return fail(KDA_ERR_UNSUPPORTED, "chunk=%d: only %d is built", chunk, kda::kPrefillChunk);
    if (L < 0) return fail(KDA_ERR_INVALID_ARG, "L=%d < 0", L);
    if (B == 0 || L == 0) return launched(cudaSuccess);
    CHECK(check_token_inputs(slot_ids, q, k, v, f_a, beta_logit, gate, out));
    const size_t need = kda::prefill_workspace_bytes(layer->num_heads, B, L);
    if (need > 0) {
        if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
            return fail(KDA_ERR_INVALID_ARG, "workspace is null or not 256-byte aligned");
        if (workspace_bytes < need)
            return fail(KDA_ERR_INVALID_ARG, "workspace_bytes=%zu < %zu", workspace_bytes, need);
    }
    const kda::RecurrentParams p = recurrent_params(layer, pool, slot_ids, B, L, q, k, v, f_a, beta_logit, gate, out);
    return launched(kda::launch_prefill(p, pool->state_dtype == KDA_STATE_BF16, workspace,
                                        static_cast<cudaStream_t>(stream)));
}

size_t kda_prefill_varlen_workspace_size(const kda_layer *layer, int32_t B, int32_t total_tokens, int32_t chunk)
{
    if (!layer || B < 0 || total_tokens < 0 || chunk != kda::kPrefillChunk) return 0;
    return kda::prefill_varlen_workspace_bytes(layer->num_heads, B, total_tokens);
}

kda_status kda_prefill_varlen(const kda_layer *layer, const kda_pool *pool, const int32_t *slot_ids,
                              int32_t B, const int32_t *cu_seqlens, int32_t total_tokens,
                              int32_t max_len, int32_t chunk, const void *q, const void *k,
                              const void *v, const void *f_a, const void *beta_logit,
                              const void *gate, void *out, void *workspace,
                              size_t workspace_bytes, void *stream)
{
    CHECK(check_layer(layer));
    CHECK(check_pool(pool));
    CHECK(check_batch(pool, B));
    if (chunk != kda::kPrefillChunk) return fail(KDA_ERR_UNSUPPORTED, "chunk=%d: only %d is built", chunk, kda::kPrefillChunk);
    if (total_tokens < 0) return fail(KDA_ERR_INVALID_ARG, "total_tokens=%d < 0", total_tokens);
    if (max_len < 0) return fail(KDA_ERR_INVALID_ARG, "max_len=%d < 0", max_len);
    if (B == 0 || total_tokens == 0) return launched(cudaSuccess);
    if (max_len == 0) return fail(KDA_ERR_INVALID_ARG, "max_len=0 with total_tokens=%d > 0", total_tokens);
    if (!cu_seqlens || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
        return fail(KDA_ERR_INVALID_ARG, "cu_seqlens is null or misaligned");
    CHECK(check_token_inputs(slot_ids, q, k, v, f_a, beta_logit, gate, out));
    const size_t need = kda::prefill_varlen_workspace_bytes(layer->num_heads, B, total_tokens);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(KDA_ERR_INVALID_ARG, "workspace is null or not 256-byte aligned");
    if (workspace_bytes < need) return fail(KDA_ERR_INVALID_ARG, "workspace_bytes=%zu < %zu", workspace_bytes, need);
    kda::RecurrentParams p = recurrent_params(layer, pool, slot_ids, B, max_len, q, k, v, f_a, beta_logit, gate, out);
    p.cu_seqlens = cu_seqlens;
    p.total_tokens = total_tokens;
    return launched(kda::launch_prefill(p, pool->state_dtype == KDA_STATE_BF16, workspace,
                                        static_cast<cudaStream_t>(stream)));
}

kda_status kda_get_error(const kda_pool *pool, int32_t *host_err, void *stream)
{
    if (!pool || !pool->err_word || !host_err) return fail(KDA_ERR_INVALID_ARG, "null argument");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, pool->err_word, sizeof v, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess && v != 0) e = cudaMemsetAsync(pool->err_word, 0, sizeof v, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "CUDA: %s", cudaGetErrorString(e));
    *host_err = v;
    g_msg[0] = '\0';
    return v ? KDA_ERR_DEVICE : KDA_OK;
}

const char *kda_status_string(kda_status s)
{
    switch (s) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
    case KDA_ERR_DEVICE: return "KDA_ERR_DEVICE";
    }
    return "KDA_ERR_UNKNOWN";
}

const char *kda_last_error(void) { return g_msg; }

int32_t kda_abi_version(void) { return KDA_ABI_VERSION; }

}  // extern "C"
