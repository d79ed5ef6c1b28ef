// Host-side launchers of the device kernels (internal to the library; the
// public entry points are in include/qlora_nf4.h).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace qlora {

// Bits of the latched device status word.
enum : unsigned {
  ST_TIMEOUT = 1u,    // a bounded wait expired
  ST_NONFINITE = 2u,  // NaN / Inf weight seen by the quantiser
};

// nf4_quant.cu
cudaError_t launch_nf4_quantize(const void* w, int w_dtype, int64_t n_elems, uint8_t* codes, float* absmax,
                                int8_t* absq, float* step, float* mean, void* ws_bins, unsigned* status,
                                uint64_t wait_ns, int num_sms, cudaStream_t s);
// Fixed scratch of the no-allocation quantise entry point (nf4_quant.cu).
int64_t noalloc_max_weights();
cudaError_t noalloc_scratch(float** absmax, void** bins);
cudaError_t launch_nf4_dequantize(const uint8_t* codes, const int8_t* absq, const float* step, const float* mean,
                                  uint16_t* out, int64_t n_elems, int num_sms, cudaStream_t s);

// lora_small.cu
size_t lora_down_workspace_bytes(int M, int K, int r, int num_sms);
// mtk [r, K] = mt^T for mt [K, r] (K % 8 == 0), plus two side jobs in the same launch:
// cvt_dst = bf16(cvt_scale * cvt_src) as in launch_lora_down, and zero_words words set to zero.
cudaError_t launch_transpose_kr(const __nv_bfloat16* mt, __nv_bfloat16* mtk, int K, int r, int num_sms, cudaStream_t s,
                                const float* cvt_src, __nv_bfloat16* cvt_dst, int64_t cvt_rows, float cvt_scale,
                                unsigned* zero, int zero_words);
// Row stride of the internal bf16 LoRA operands sT / sU ([rows, r] padded with
// zero columns): r rounded up to a multiple of 8, so every row starts on a
// 16-byte boundary as TMA requires.
__host__ __device__ inline int lora_ld(int r) { return (r + 7) & ~7; }
// out = in . mt^T with mt either [r, K] (mt_kmajor) or [K, r], by at most
// max_ctas persistent CTAs: out_f32 [M, r], out_bf16 = bf16(scale out) [M, lora_ld(r)];
// optional side job cvt_dst = bf16(cvt_scale * cvt_src) for the cvt_rows x r
// matrix cvt_src into cvt_dst [cvt_rows, lora_ld(r)], in the same launch.
cudaError_t launch_lora_down(const __nv_bfloat16* in, const __nv_bfloat16* mt, int mt_kmajor, int M, int K, int r,
                             float scale, float* out_f32, __nv_bfloat16* out_bf16, void* ws, int max_ctas,
                             cudaStream_t s, const float* cvt_src = nullptr, __nv_bfloat16* cvt_dst = nullptr,
                             int64_t cvt_rows = 0, float cvt_scale = 1.0f, float t_scale = 1.0f);
// The same product for r <= 16 with k split over a cluster of up to 4 CTAs per 64-row block (one
// wave of row blocks at most); lora_down_ks_plan says whether a shape takes it and its split.
bool lora_down_ks_plan(int M, int K, int r, int num_sms, int* splits, int* chunks_per_split);
cudaError_t launch_lora_down_ks(const __nv_bfloat16* in, const __nv_bfloat16* mt, int mt_kmajor, int M, int K, int r,
                                float scale, float* out_f32, __nv_bfloat16* out_bf16, int num_sms, cudaStream_t s,
                                const float* cvt_src = nullptr, __nv_bfloat16* cvt_dst = nullptr,
                                int64_t cvt_rows = 0, float cvt_scale = 1.0f, float t_scale = 1.0f);
cudaError_t launch_silu_mul_fwd(const uint16_t* g, const uint16_t* u, uint16_t* h, int64_t n, int num_sms,
                                cudaStream_t s);
cudaError_t launch_silu_mul_bwd(const uint16_t* dh, const uint16_t* g, const uint16_t* u, uint16_t* dg, uint16_t* du,
                                int64_t n, int num_sms, cudaStream_t s);

// qgemm.cu
struct Nf4Dev {
  const uint8_t* codes;
  const int8_t* absq;
  const float* step;
  const float* mean;
  int64_t n, k;
};

// Forward / decode: Y[M, N] = X[M, K] deq(W)^T + sT[M, r] B[N, r]^T   (sT = bf16(s * X A^T))
size_t fwd_gemm_workspace_bytes(int M, int N, int K, int num_sms);
cudaError_t launch_fwd_gemm(const __nv_bfloat16* x, int M, const Nf4Dev& w, const __nv_bfloat16* st,
                            const __nv_bfloat16* lora_b, int r, __nv_bfloat16* y, void* ws, unsigned* status,
                            uint64_t wait_ns, int num_sms, cudaStream_t s);

// Backward dX[M, K] (+)= dY[M, N] deq(W) + sU[M, r] A[r, K]   (sU = bf16(s * dY B))
// with_lora = 0: the LoRA k steps are left out (dX = dY deq(W) only; the dropout path adds its
// masked LoRA term separately).
// ws: bwd_gemm_workspace_bytes (fp32 partials of the split n blocks and per-tile counters).
size_t bwd_gemm_workspace_bytes(int M, int N, int K, int num_sms);
cudaError_t launch_bwd_dx_gemm(const __nv_bfloat16* dy, int M, const Nf4Dev& w, const __nv_bfloat16* su,
                               const __nv_bfloat16* lora_a, int r, __nv_bfloat16* dx, int accumulate, void* ws,
                               unsigned* status, uint64_t wait_ns, int num_sms, cudaStream_t s, int with_lora = 1);

// LoRA gradients: dA[r, K] (+)= sU^T X   and   dB[N, r] (+)= dY^T sT
size_t lora_grads_workspace_bytes(int M, int N, int K, int r, int num_sms);
cudaError_t launch_lora_grads(const __nv_bfloat16* x, const __nv_bfloat16* dy, const __nv_bfloat16* su,
                              const __nv_bfloat16* st, int M, int N, int K, int r, float* da, float* db,
                              int accum_da, int accum_db, void* ws, unsigned* status, uint64_t wait_ns, int max_ctas,
                              cudaStream_t s, float da_scale = 1.0f);
// CTA-pair versions of both GEMMs (qgemm_pair.cu), used for M > 256 tokens.
bool use_pair_gemm(int M);
int fwd_pair_ctas(int M, int N);
int bwd_pair_ctas(int M, int K);
cudaError_t launch_fwd_gemm_pair(const __nv_bfloat16* x, int M, const Nf4Dev& w, const __nv_bfloat16* st,
                                 const __nv_bfloat16* lora_b, int r, __nv_bfloat16* y, unsigned* status,
                                 uint64_t wait_ns, cudaStream_t s);
cudaError_t launch_bwd_gemm_pair(const __nv_bfloat16* dy, int M, const Nf4Dev& w, const __nv_bfloat16* su,
                                 const __nv_bfloat16* lora_a, int r, __nv_bfloat16* dx, int accumulate,
                                 unsigned* status, uint64_t wait_ns, cudaStream_t s, int with_lora = 1);
// Low-rank combinations (nf4_merge.cu).
// out[n, k] = bf16(deq(W) + scale * B A), the B A sum a float32 FMA chain in j order.
cudaError_t launch_nf4_merge(const Nf4Dev& w, const __nv_bfloat16* lora_a, const __nv_bfloat16* lora_b, int r,
                             float scale, __nv_bfloat16* out, cudaStream_t s);
// out[n, k] = (W - deq(sub)) + coef * B A in float32 (sub may be null; r may be 0).
cudaError_t launch_lowrank_update(const void* dense, int dense_bf16, const Nf4Dev* sub, const __nv_bfloat16* lora_a,
                                  const __nv_bfloat16* lora_b, int r, float coef, float* out, int64_t n, int64_t k,
                                  cudaStream_t s);
// AdamW on a list of tensors in one launch (adamw.cu).
struct AdamwTensor {
  float* master;          // float32 weights (updated)
  __nv_bfloat16* param;   // bf16 copy the kernels read (written; may be null)
  const float* grad;
  float* exp_avg;
  float* exp_avg_sq;
  int64_t numel;
};
struct AdamwHyper {
  float decay, beta1, omb1, beta2, omb2, step_size, bc2_sqrt, eps;
};
// The float32 factors of step `step` (1-based), formed in double precision.
AdamwHyper adamw_hyper(double lr, double beta1, double beta2, double eps, double weight_decay, int64_t step);
cudaError_t launch_adamw(const AdamwTensor* tensors, int count, const AdamwHyper& h, int num_sms, cudaStream_t s);
// LoRA dropout (dropout.cu): Philox4x32-10 keep mask, one bit per element of an [m, k] input
// (n_elems % 64 == 0), and x_drop = x * mask (bf16).
cudaError_t launch_dropout_mask(uint64_t seed, uint64_t offset, int64_t n_elems, float p, uint8_t* mask, int num_sms,
                                cudaStream_t s);
cudaError_t launch_dropout_apply(const uint16_t* x, const uint8_t* mask, uint16_t* x_drop, int64_t n_elems, int num_sms,
                                 cudaStream_t s);
// dx[m, k] = bf16(dx + (keep(m, k) ? coef * sum_j su[m, j] a[j, k] : 0)), su with row stride lora_ld(r)
// (nf4_merge.cu): the LoRA term of dX under dropout.
cudaError_t launch_dropout_lora_dx(__nv_bfloat16* dx, const __nv_bfloat16* su, const __nv_bfloat16* lora_a,
                                   const uint8_t* mask, int M, int K, int r, float coef, cudaStream_t s);
// 2-D bf16 tensor map, 128-byte swizzle, zero fill outside [outer x inner] (qgemm.cu).
bool make_tensor_map_bf16_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch,
                             uint32_t box_inner, uint32_t box_outer);
// Forward LoRA down-projection beside the pair GEMM (lora_side.cu), 1 <= r <= 64:
// T = X A^T -> t_save, sT = bf16(s T), by at most max_ctas CTAs.
bool lora_side_supported(int r);
// Backward U = dY B beside the dX GEMM: dY [M, N], bt = B^T [r, N] (N % 64 == 0), su = bf16(scale U)
// [M, lora_ld(r)]; k is split over CTAs (ws: lora_side_bwd_workspace_bytes; its counter words,
// lora_side_bwd_counters, must be zero at launch and are zero again afterwards).
size_t lora_side_bwd_workspace_bytes(int M, int K, int r, int num_sms);
unsigned* lora_side_bwd_counters(void* ws, int M, int K, int r, int num_sms);
cudaError_t launch_lora_side_bwd(const __nv_bfloat16* dy, const __nv_bfloat16* bt, int M, int N, int r, float scale,
                                 __nv_bfloat16* su, void* ws, int num_sms, unsigned* status, uint64_t wait_ns,
                                 cudaStream_t s);

cudaError_t launch_lora_side_fwd(const __nv_bfloat16* x, const __nv_bfloat16* lora_a, int M, int K, int r, float scale,
                                 float* t_save, __nv_bfloat16* st, int max_ctas, unsigned* status, uint64_t wait_ns,
                                 cudaStream_t s, float t_scale = 1.0f);
// Grid sizes of the GEMMs and the SMs they leave idle (budget for side kernels).
int fwd_gemm_ctas(int M, int N, int K, int num_sms);
int bwd_gemm_ctas(int M, int N, int K, int num_sms);
int idle_sms_beside(int gemm_ctas, int num_sms);

// Grouped small-token forward (decode.cu): one problem of the list.
struct GroupedProblem {
  const __nv_bfloat16* x;       // [m, k], 1 <= m <= 16
  Nf4Dev w;                     // [n, k]
  const __nv_bfloat16* lora_a;  // [r, k]
  const __nv_bfloat16* lora_b;  // [n, r]
  int m, r;                     // 1 <= r <= 128
  float alpha;
  __nv_bfloat16* y;             // [m, n]
  float* t_save;                // [m, r] or null
};
// Problems per launch; a longer list goes out in several launches.
int decode_max_problems();
size_t decode_workspace_bytes(const GroupedProblem* probs, int count, int num_sms);
// One launch for the whole list (count <= decode_max_problems()).  The workspace's counters
// must be zero before the first call; every call leaves them zero.
cudaError_t launch_decode(const GroupedProblem* probs, int count, void* ws, unsigned* status, uint64_t wait_ns,
                          int num_sms, cudaStream_t s);

// Bounded-wait self test: one CTA waits on an mbarrier nothing arrives on.
cudaError_t launch_wait_selftest(unsigned* status, uint64_t wait_ns, cudaStream_t s);

const char* tensor_map_error();

}  // namespace qlora
