// internal.h -- launchers behind the C ABI (fp8rl.h).  Arguments reaching these
// functions have been validated by abi.cu; the launchers only size grids and
// launch on the given stream.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fp8rl {

constexpr int kBlk = 128;          // weight block edge and activation group length
constexpr int kMaxGroup = 256;        // tensors per grouped requant launch
constexpr int64_t kInt8MaxK = 32768;  // row length held in registers by the INT8 quantizer

struct WeightDesc {
    const uint16_t* W;
    uint8_t* Wq;
    float* Ws;
    int64_t N, K, ldw;
};

cudaError_t launch_quant_weight_block(const WeightDesc* d, int n, cudaStream_t st);
cudaError_t launch_quant_act_group(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                                   uint8_t* Xq, float* Xs, cudaStream_t st);
cudaError_t launch_quant_int8_rows(const uint16_t* A, int64_t R, int64_t K, int64_t lda,
                                   int8_t* Q, float* S, cudaStream_t st);

// FP8 KV-cache per-tensor quant: one cooperative launch over a header word and
// kv_partials(R, C) 8-byte slots when every slice's CTA fits at once, else three
// launches over kv_partials(R, C) 32-bit words placed after the header;
// `partial` is 8-byte aligned and holds (kv_partials(R, C) + 1) * 8 bytes.
int64_t kv_partials(int64_t R, int64_t C);
cudaError_t launch_quant_kv_tensor(const uint16_t* X, int64_t R, int64_t C, int64_t ld, uint8_t* Xq,
                                   float* scale, uint32_t* partial, cudaStream_t st);
cudaError_t launch_quant_kv_with_scale(const uint16_t* X, int64_t R, int64_t C, int64_t ld,
                                       const float* scale, uint8_t* Xq, cudaStream_t st);
// The same with the partial maxima in a library-owned device array (no workspace).
int64_t kv_noalloc_max_values();
cudaError_t launch_quant_kv_tensor_noalloc(const uint16_t* X, int64_t R, int64_t C, int64_t ld,
                                           uint8_t* Xq, float* scale, cudaStream_t st);

// Token-level TIS/MIS weights and statistics (two launches, partial records in `ws`).
int64_t rollout_is_partials(int64_t n);
int64_t rollout_is_max_partials(int64_t n);
size_t rollout_is_partial_bytes();
cudaError_t launch_rollout_is(const float* lt, const float* lr, const uint8_t* mask, int64_t n,
                              float log_clip, int mode, float* w, double* stats, void* ws,
                              cudaStream_t st);

// Per-token KL between two logit matrices (two launches, partial records in `ws`).
int kl_chunks(int64_t V);
size_t kl_partial_bytes();
cudaError_t launch_logits_kl(const uint16_t* P, int64_t ldp, const uint16_t* Q, int64_t ldq, int64_t M,
                             int64_t V, float* kl, void* ws, cudaStream_t st);

// FP8 block-scaled GEMM: dispatch by M (tcgen05 decode kernel for M <= 256).
// weights_stable: the kernel immediately preceding the call in the stream did
// not write Wq, so small weights may start streaming before the dependency wait.
cudaError_t launch_gemm_fp8_decode(const uint8_t* Xq, const float* Xs, const uint8_t* Wq,
                                   const float* Ws, int64_t M, int64_t N, int64_t K, uint16_t* Y,
                                   int64_t ldy, void* ws, size_t ws_bytes, bool weights_stable,
                                   cudaStream_t st);
size_t decode_workspace_bytes(int64_t M, int64_t N, int64_t K);
int decode_kernel_count(int64_t M, int64_t N, int64_t K, size_t ws_bytes);
int gemm_fp8_kernel_count(int64_t M, int64_t N, int64_t K, size_t ws_bytes);
int gemm_int8_kernel_count(int64_t M, int64_t N, int64_t K, size_t ws_bytes);
int int8_prefill_kernel_count(int64_t M, int64_t N, int64_t K);
// Grouped (mixture-of-experts) form of the decode kernel: experts' weights
// stacked [E*N][K], token rows grouped by expert at offs[0..E] (device).
cudaError_t launch_gemm_fp8_grouped(const uint8_t* Xq, const float* Xs, const uint8_t* Wq, const float* Ws,
                                    const int32_t* offs, int64_t E, int64_t T, int64_t N, int64_t K,
                                    int64_t max_rows, uint16_t* Y, int64_t ldy, cudaStream_t st);
size_t gemm_fp8_workspace_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemm_fp8(const uint8_t* Xq, const float* Xs, const uint8_t* Wq,
                            const float* Ws, int64_t M, int64_t N, int64_t K, uint16_t* Y,
                            int64_t ldy, void* ws, size_t ws_bytes, bool weights_stable, cudaStream_t st);

// INT8 GEMM: exact integer arithmetic on the fp16 tensor path (tcgen05).
cudaError_t launch_gemm_int8_tc(const int8_t* Xq, const float* Xs, const int8_t* Wq, const float* Ws,
                                int64_t M, int64_t N, int64_t K, uint16_t* Y, int64_t ldy, int32_t* acc,
                                cudaStream_t st);
// INT8 GEMM.
size_t gemm_int8_workspace_bytes(int64_t M, int64_t N, int64_t K);
// Large-batch INT8 path: int8 -> fp16 copies in the workspace, then a 128 x 256
// tile fp16 tcgen05 GEMM with exact int32 accumulation.
bool int8_prefill_applies(int64_t M, int64_t N, int64_t K);
size_t int8_prefill_workspace_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemm_int8_prefill(const int8_t* Xq, const float* Xs, const int8_t* Wq, const float* Ws,
                                     int64_t M, int64_t N, int64_t K, uint16_t* Y, int64_t ldy, int32_t* acc,
                                     void* ws, cudaStream_t st);
// fp16 copy of n int8 codes (exact), n % 16 == 0.
cudaError_t launch_int8_to_f16(const int8_t* src, int64_t n, uint16_t* dst, cudaStream_t st);
// Mid-size batches: weight blocks in TMEM, 256-token tiles of an fp16 copy of X
// (in the workspace, with the int32 partials of a K split).
size_t int8_t256_workspace_bytes(int64_t M, int64_t N, int64_t K);
int int8_t256_kernel_count(int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemm_int8_t256(const int8_t* Xq, const float* Xs, const int8_t* Wq, const float* Ws,
                                  int64_t M, int64_t N, int64_t K, uint16_t* Y, int64_t ldy, int32_t* acc,
                                  void* ws, cudaStream_t st);
cudaError_t launch_gemm_int8(const int8_t* Xq, const float* Xs, const int8_t* Wq,
                             const float* Ws, int64_t M, int64_t N, int64_t K, uint16_t* Y,
                             int64_t ldy, int32_t* acc, void* ws, size_t ws_bytes,
                             cudaStream_t st);

// The linear layer from bf16 activations: the activation quantizer, then the GEMM.
size_t linear_codes_bytes(int64_t M, int64_t K);
size_t linear_workspace_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t launch_linear_fp8(const uint16_t* X, int64_t ldx, const uint8_t* Wq, const float* Ws, int64_t M,
                              int64_t N, int64_t K, uint16_t* Y, int64_t ldy, uint8_t* Xq_out,
                              float* Xs_out, void* ws, cudaStream_t st);

// Device-side record of a bounded wait that ran out (0 = none).
cudaError_t read_and_clear_device_error(uint32_t* word);
// Address of that word on the current device (passed to kernels that wait).
uint32_t* device_error_word();

// TMA map of a row-major byte matrix [rows][cols] (row pitch `pitch` bytes),
// boxes of 128 columns x box_rows rows, 128-byte swizzle, zero fill out of range.
bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t pitch,
                  uint32_t box_rows);
// TMA map of a row-major bf16 matrix [rows][cols] (row pitch in elements) for
// stores of box_cols x box_rows boxes with the 128-byte swizzle (box_cols = 64).
bool make_tmap_bf16_store(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                          uint64_t pitch_elems, uint32_t box_cols, uint32_t box_rows);
// TMA map of a row-major fp32 matrix [rows][cols] (row pitch in elements) for
// stores of box_cols x box_rows boxes with the 128-byte swizzle (box_cols = 32).
bool make_tmap_f32_store(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                         uint64_t pitch_elems, uint32_t box_cols, uint32_t box_rows);
// fp16 [rows][cols] row-major (cols % 8 == 0), loaded in boxes of box_rows x 64
// with the 128-byte swizzle (one UMMA K-major atom of fp16).
bool make_tmap_f16_load(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);
int num_sms();
bool decode_supported(int64_t K);
bool decode_fits(int64_t M, int64_t N, int64_t K, size_t ws_bytes);
double decode_cost_us(int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemm_fp8_prefill(const uint8_t* Xq, const float* Xs, const uint8_t* Wq,
                                    const float* Ws, int64_t M, int64_t N, int64_t K, uint16_t* Y,
                                    int64_t ldy, void* ws, size_t ws_bytes, cudaStream_t st);

}  // namespace fp8rl
