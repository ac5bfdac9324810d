// abi.cu -- the extern "C" boundary declared in include/fp8rl.h: synchronous
// argument validation, then one launch (or a few) on the caller's stream.
#include <vector>

#include "fp8rl.h"
#include "internal.h"


namespace {

using namespace fp8rl;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? FP8RL_OK : FP8RL_ERR_CUDA; }

// Common checks of a bf16 [R][ld] source with row length K (K a multiple of 128).
int check_bf16_src(const uint16_t* A, int64_t R, int64_t K, int64_t ld, bool need_k128) {
    if (R < 0 || K <= 0 || ld < K) return FP8RL_ERR_SHAPE;
    if (need_k128 && K % kBlk) return FP8RL_ERR_SHAPE;
    if (!need_k128 && K % 16) return FP8RL_ERR_SHAPE;
    if (R > 0 && !A) return FP8RL_ERR_NULL;
    if (!aligned16(A) || (ld * 2) % 16) return FP8RL_ERR_ALIGN;
    return FP8RL_OK;
}

int check_weight_desc(const fp8rl_wdesc& d) {
    if (d.N < 0 || d.N % kBlk) return FP8RL_ERR_SHAPE;
    int rc = check_bf16_src(d.W, d.N, d.K, d.ldw, true);
    if (rc) return rc;
    if (d.N > 0 && (!d.Wq || !d.Ws)) return FP8RL_ERR_NULL;
    if (!aligned16(d.Wq) || !aligned4(d.Ws)) return FP8RL_ERR_ALIGN;
    return FP8RL_OK;
}

int check_gemm_common(const void* Xq, const float* Xs, const void* Wq, const float* Ws,
                      int64_t M, int64_t N, int64_t K, const uint16_t* Y, int64_t ldy) {
    if (M < 0 || N <= 0 || K <= 0 || N % kBlk || K % kBlk || ldy < N) return FP8RL_ERR_SHAPE;
    if (!Wq || !Ws) return FP8RL_ERR_NULL;
    if (M > 0 && (!Xq || !Xs || !Y)) return FP8RL_ERR_NULL;
    if (!aligned16(Xq) || !aligned16(Wq) || !aligned16(Y) || !aligned4(Xs) || !aligned4(Ws))
        return FP8RL_ERR_ALIGN;
    if ((ldy * 2) % 16) return FP8RL_ERR_ALIGN;
    return FP8RL_OK;
}

}  // namespace

extern "C" {

const char* fp8rl_status_string(int status) {
    switch (status) {
        case FP8RL_OK: return "FP8RL_OK";
        case FP8RL_ERR_NULL: return "FP8RL_ERR_NULL: required pointer is NULL";
        case FP8RL_ERR_SHAPE: return "FP8RL_ERR_SHAPE: invalid size or leading dimension";
        case FP8RL_ERR_ALIGN: return "FP8RL_ERR_ALIGN: pointer or row pitch not 16-byte aligned";
        case FP8RL_ERR_WORKSPACE: return "FP8RL_ERR_WORKSPACE: workspace too small";
        case FP8RL_ERR_CUDA: return "FP8RL_ERR_CUDA: CUDA runtime reported an error";
        case FP8RL_ERR_UNSUPPORTED: return "FP8RL_ERR_UNSUPPORTED: size above a documented limit";
        case FP8RL_ERR_TIMEOUT: return "FP8RL_ERR_TIMEOUT: a bounded device-side wait ran out";
        case FP8RL_ERR_DEVICE: return "FP8RL_ERR_DEVICE: a device-side check of the data failed";
        default: return "FP8RL_ERR_UNKNOWN";
    }
}

int fp8rl_abi_version(void) { return FP8RL_ABI_VERSION; }

int fp8rl_quant_weight_block(const uint16_t* W, int64_t N, int64_t K, int64_t ldw, uint8_t* Wq,
                             float* Ws, void* stream) {
    fp8rl_wdesc d{W, Wq, Ws, N, K, ldw};
    return fp8rl_quant_weight_block_grouped(&d, 1, stream);
}

int fp8rl_quant_weight_block_grouped(const fp8rl_wdesc* descs, int n, void* stream) {
    if (n < 0) return FP8RL_ERR_SHAPE;
    if (n > 0 && !descs) return FP8RL_ERR_NULL;
    std::vector<WeightDesc> v;
    v.reserve(n);
    for (int i = 0; i < n; ++i) {
        int rc = check_weight_desc(descs[i]);
        if (rc) return rc;
        v.push_back({descs[i].W, descs[i].Wq, descs[i].Ws, descs[i].N, descs[i].K, descs[i].ldw});
    }
    return cuda_status(launch_quant_weight_block(v.data(), n, as_stream(stream)));
}

int fp8rl_quant_act_group(const uint16_t* X, int64_t M, int64_t K, int64_t ldx, uint8_t* Xq,
                          float* Xs, void* stream) {
    int rc = check_bf16_src(X, M, K, ldx, true);
    if (rc) return rc;
    if (M > 0 && (!Xq || !Xs)) return FP8RL_ERR_NULL;
    if (!aligned16(Xq) || !aligned4(Xs)) return FP8RL_ERR_ALIGN;
    if (M > 65535LL * 16) return FP8RL_ERR_UNSUPPORTED;
    return cuda_status(launch_quant_act_group(X, M, K, ldx, Xq, Xs, as_stream(stream)));
}

size_t fp8rl_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    return gemm_fp8_workspace_bytes(M, N, K);
}

int fp8rl_gemm_kernel_count(int64_t M, int64_t N, int64_t K, size_t workspace_bytes) {
    if (M < 0 || N <= 0 || K <= 0 || N % kBlk || K % kBlk) return -FP8RL_ERR_SHAPE;
    return gemm_fp8_kernel_count(M, N, K, workspace_bytes);
}

int fp8rl_gemm_w8a8_block_ex(const uint8_t* Xq, const float* Xs, const uint8_t* Wq, const float* Ws,
                             int64_t M, int64_t N, int64_t K, uint16_t* Y, int64_t ldy,
                             void* workspace, size_t workspace_bytes, unsigned flags, void* stream) {
    int rc = check_gemm_common(Xq, Xs, Wq, Ws, M, N, K, Y, ldy);
    if (rc) return rc;
    if (flags & ~(unsigned)FP8RL_GEMM_WEIGHTS_STABLE) return FP8RL_ERR_UNSUPPORTED;
    if (M > 65535LL * 32) return FP8RL_ERR_UNSUPPORTED;
    if (!aligned16(workspace)) return FP8RL_ERR_ALIGN;
    if (M == 0) return FP8RL_OK;
    // less workspace than the query only gives up split-K (see the header)
    return cuda_status(launch_gemm_fp8(Xq, Xs, Wq, Ws, M, N, K, Y, ldy, workspace,
                                       workspace ? workspace_bytes : 0,
                                       (flags & FP8RL_GEMM_WEIGHTS_STABLE) != 0, as_stream(stream)));
}

int fp8rl_gemm_w8a8_block(const uint8_t* Xq, const float* Xs, const uint8_t* Wq, const float* Ws,
                          int64_t M, int64_t N, int64_t K, uint16_t* Y, int64_t ldy,
                          void* workspace, size_t workspace_bytes, void* stream) {
    return fp8rl_gemm_w8a8_block_ex(Xq, Xs, Wq, Ws, M, N, K, Y, ldy, workspace, workspace_bytes, 0u, stream);
}

int fp8rl_gemm_w8a8_block_grouped(const uint8_t* Xq, const float* Xs, const uint8_t* Wq,
                                  const float* Ws, const int32_t* expert_offsets, int64_t E,
                                  int64_t T, int64_t N, int64_t K, int64_t max_tokens_per_expert,
                                  uint16_t* Y, int64_t ldy, void* stream) {
    if (E < 1 || T < 0) return FP8RL_ERR_SHAPE;
    int rc = check_gemm_common(Xq, Xs, Wq, Ws, T, N, K, Y, ldy);
    if (rc) return rc;
    if (!expert_offsets) return FP8RL_ERR_NULL;
    if (!aligned4(expert_offsets)) return FP8RL_ERR_ALIGN;
    if (T > 0 && (max_tokens_per_expert < 1 || max_tokens_per_expert > T)) return FP8RL_ERR_SHAPE;
    if (!decode_supported(K) || E * (N / kBlk) > 65535 || T > 0x7FFFFFFFLL) return FP8RL_ERR_UNSUPPORTED;
    if (T == 0) return FP8RL_OK;
    return cuda_status(launch_gemm_fp8_grouped(Xq, Xs, Wq, Ws, expert_offsets, E, T, N, K,
                                               max_tokens_per_expert, Y, ldy, as_stream(stream)));
}

size_t fp8rl_linear_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    return linear_workspace_bytes(M, N, K);
}

int fp8rl_linear_kernel_count(int64_t M, int64_t N, int64_t K, size_t workspace_bytes, int want_codes) {
    (void)want_codes;                                   // the same kernels either way
    if (M < 0 || N <= 0 || K <= 0 || N % kBlk || K % kBlk) return -FP8RL_ERR_SHAPE;
    if (M == 0) return 0;
    const size_t g = gemm_fp8_workspace_bytes(M, N, K);
    const size_t gws = (g && workspace_bytes >= linear_workspace_bytes(M, N, K)) ? g : 0;
    return 1 + gemm_fp8_kernel_count(M, N, K, gws);
}

int fp8rl_linear_w8a8_block(const uint16_t* X, int64_t ldx, const uint8_t* Wq, const float* Ws,
                            int64_t M, int64_t N, int64_t K, uint16_t* Y, int64_t ldy,
                            uint8_t* Xq_or_null, float* Xs_or_null, void* workspace,
                            size_t workspace_bytes, void* stream) {
    int rc = check_bf16_src(X, M, K, ldx, true);
    if (rc) return rc;
    if (N <= 0 || N % kBlk || ldy < N) return FP8RL_ERR_SHAPE;
    if (!Wq || !Ws || (M > 0 && !Y)) return FP8RL_ERR_NULL;
    if ((Xq_or_null == nullptr) != (Xs_or_null == nullptr)) return FP8RL_ERR_NULL;
    if (!aligned16(Wq) || !aligned16(Y) || !aligned4(Ws) || (ldy * 2) % 16) return FP8RL_ERR_ALIGN;
    if (!aligned16(Xq_or_null) || !aligned4(Xs_or_null) || !aligned16(workspace)) return FP8RL_ERR_ALIGN;
    if (M > 65535LL * 16) return FP8RL_ERR_UNSUPPORTED;
    const size_t need = fp8rl_linear_workspace_bytes(M, N, K);
    if (workspace_bytes < need || (need && !workspace)) return FP8RL_ERR_WORKSPACE;
    if (M == 0) return FP8RL_OK;
    return cuda_status(launch_linear_fp8(X, ldx, Wq, Ws, M, N, K, Y, ldy, Xq_or_null, Xs_or_null,
                                         workspace, as_stream(stream)));
}

int int8rl_quant_weight_channel(const uint16_t* W, int64_t N, int64_t K, int64_t ldw, int8_t* Wq,
                                float* Ws, void* stream) {
    int rc = check_bf16_src(W, N, K, ldw, true);
    if (rc) return rc;
    if (K > kInt8MaxK) return FP8RL_ERR_UNSUPPORTED;
    if (N > 0 && (!Wq || !Ws)) return FP8RL_ERR_NULL;
    if (!aligned16(Wq) || !aligned4(Ws)) return FP8RL_ERR_ALIGN;
    return cuda_status(launch_quant_int8_rows(W, N, K, ldw, Wq, Ws, as_stream(stream)));
}

int int8rl_quant_act_token(const uint16_t* X, int64_t M, int64_t K, int64_t ldx, int8_t* Xq,
                           float* Xs, void* stream) {
    return int8rl_quant_weight_channel(X, M, K, ldx, Xq, Xs, stream);
}

size_t int8rl_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    return gemm_int8_workspace_bytes(M, N, K);
}

int int8rl_gemm_kernel_count(int64_t M, int64_t N, int64_t K, size_t workspace_bytes) {
    if (M < 0 || N <= 0 || K <= 0 || N % kBlk || K % kBlk) return -FP8RL_ERR_SHAPE;
    return gemm_int8_kernel_count(M, N, K, workspace_bytes);
}

int int8rl_gemm_w8a8(const int8_t* Xq, const float* Xs, const int8_t* Wq, const float* Ws,
                     int64_t M, int64_t N, int64_t K, uint16_t* Y, int64_t ldy,
                     int32_t* acc_or_null, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_gemm_common(Xq, Xs, Wq, Ws, M, N, K, Y, ldy);
    if (rc) return rc;
    if (K > 133143) return FP8RL_ERR_UNSUPPORTED;       // 127^2 * K must stay below 2^31
    if (M > 65535LL * 32) return FP8RL_ERR_UNSUPPORTED;
    if (acc_or_null && (reinterpret_cast<uintptr_t>(acc_or_null) & 7u)) return FP8RL_ERR_ALIGN;
    if (!aligned16(workspace)) return FP8RL_ERR_ALIGN;
    if (M == 0) return FP8RL_OK;
    // less workspace than the query only gives up the large-batch path (see the header)
    return cuda_status(launch_gemm_int8(Xq, Xs, Wq, Ws, M, N, K, Y, ldy, acc_or_null, workspace,
                                        workspace ? workspace_bytes : 0, as_stream(stream)));
}

static int check_kv(const uint16_t* KV, int64_t R, int64_t C, int64_t ld, const uint8_t* KVq) {
    if (R < 0 || C <= 0 || C % 8 || ld < C) return FP8RL_ERR_SHAPE;
    if (R > 0 && (!KV || !KVq)) return FP8RL_ERR_NULL;
    if (!aligned16(KV) || !aligned16(KVq) || (ld * 2) % 16) return FP8RL_ERR_ALIGN;
    return FP8RL_OK;
}

size_t fp8rl_kv_workspace_bytes(int64_t R, int64_t C) {
    if (R <= 0 || C <= 0) return 0;
    return (size_t)(kv_partials(R, C) + 1) * sizeof(uint64_t);   // the header word + one 8-byte slot per slice
}

int fp8rl_quant_kv_tensor(const uint16_t* KV, int64_t R, int64_t C, int64_t ld, uint8_t* KVq,
                          float* scale, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_kv(KV, R, C, ld, KVq);
    if (rc) return rc;
    if (!scale) return FP8RL_ERR_NULL;
    if (!aligned4(scale) || !aligned8(workspace)) return FP8RL_ERR_ALIGN;
    const size_t need = fp8rl_kv_workspace_bytes(R, C);
    if (workspace_bytes < need || (need && !workspace)) return FP8RL_ERR_WORKSPACE;
    return cuda_status(launch_quant_kv_tensor(KV, R, C, ld, KVq, scale,
                                              static_cast<uint32_t*>(workspace), as_stream(stream)));
}

int fp8rl_quant_kv_with_scale(const uint16_t* KV, int64_t R, int64_t C, int64_t ld,
                              const float* scale, uint8_t* KVq, void* stream) {
    int rc = check_kv(KV, R, C, ld, KVq);
    if (rc) return rc;
    if (!scale) return FP8RL_ERR_NULL;
    if (!aligned4(scale)) return FP8RL_ERR_ALIGN;
    return cuda_status(launch_quant_kv_with_scale(KV, R, C, ld, scale, KVq, as_stream(stream)));
}

size_t fp8rl_rollout_is_workspace_bytes(int64_t n) {
    if (n <= 0) return 0;
    return 8 + (size_t)rollout_is_max_partials(n) * rollout_is_partial_bytes();   // header word + records
}

int fp8rl_rollout_is_weights(const float* logp_train, const float* logp_rollout, const uint8_t* mask,
                             int64_t n, float log_clip, int mode, float* weights, double* stats,
                             void* workspace, size_t workspace_bytes, void* stream) {
    if (n < 0 || (mode != FP8RL_IS_TRUNCATE && mode != FP8RL_IS_MASK)) return FP8RL_ERR_SHAPE;
    if (!stats || (n > 0 && (!logp_train || !logp_rollout || !weights))) return FP8RL_ERR_NULL;
    if (!aligned4(logp_train) || !aligned4(logp_rollout) || !aligned4(weights) ||
        (reinterpret_cast<uintptr_t>(stats) & 7u) || (reinterpret_cast<uintptr_t>(workspace) & 7u))
        return FP8RL_ERR_ALIGN;
    const size_t need = fp8rl_rollout_is_workspace_bytes(n);
    if (workspace_bytes < need || (need && !workspace)) return FP8RL_ERR_WORKSPACE;
    return cuda_status(launch_rollout_is(logp_train, logp_rollout, mask, n, log_clip, mode, weights,
                                         stats, workspace, as_stream(stream)));
}

size_t fp8rl_logits_kl_workspace_bytes(int64_t M, int64_t V) {
    if (M <= 0 || V <= 0) return 0;
    return (size_t)M * (size_t)kl_chunks(V) * kl_partial_bytes();
}

int fp8rl_logits_kl(const uint16_t* P, int64_t ldp, const uint16_t* Q, int64_t ldq, int64_t M,
                    int64_t V, float* kl, void* workspace, size_t workspace_bytes, void* stream) {
    if (M < 0 || V < 1 || ldp < V || ldq < V) return FP8RL_ERR_SHAPE;
    if (M > 0 && (!P || !Q || !kl)) return FP8RL_ERR_NULL;
    if (!aligned16(P) || !aligned16(Q) || (ldp * 2) % 16 || (ldq * 2) % 16 || !aligned4(kl) ||
        !aligned16(workspace))
        return FP8RL_ERR_ALIGN;
    if (M > 65535) return FP8RL_ERR_UNSUPPORTED;
    const size_t need = fp8rl_logits_kl_workspace_bytes(M, V);
    if (workspace_bytes < need || (need && !workspace)) return FP8RL_ERR_WORKSPACE;
    if (M == 0) return FP8RL_OK;
    return cuda_status(launch_logits_kl(P, ldp, Q, ldq, M, V, kl, workspace, as_stream(stream)));
}

int fp8rl_quant_kv_tensor_noalloc(const uint16_t* KV, int64_t R, int64_t C, int64_t ld, uint8_t* KVq,
                                  float* scale, void* stream) {
    int rc = check_kv(KV, R, C, ld, KVq);
    if (rc) return rc;
    if (!scale) return FP8RL_ERR_NULL;
    if (!aligned4(scale)) return FP8RL_ERR_ALIGN;
    if (R > 0 && R > kv_noalloc_max_values() / C) return FP8RL_ERR_UNSUPPORTED;   // R * C above the limit
    return cuda_status(launch_quant_kv_tensor_noalloc(KV, R, C, ld, KVq, scale, as_stream(stream)));
}

int fp8rl_check_device_error(uint32_t* detail) {
    uint32_t w = 0;
    cudaError_t e = read_and_clear_device_error(&w);
    if (detail) *detail = w;
    if (e != cudaSuccess) return FP8RL_ERR_CUDA;
    if (!w) return FP8RL_OK;
    return (w & 0xFFFFu) == 2u ? FP8RL_ERR_DEVICE : FP8RL_ERR_TIMEOUT;
}

}  // extern "C"
