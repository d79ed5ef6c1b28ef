// AdamW step on the LoRA matrices, for optimizer state in paged (managed) memory.
//
// The pages: P1 tutorial "QLoRA: fine-tuning 7B on a 24 GB card", section 3.3
// (optim="paged_adamw_8bit"), tbr8.org "QLoRA on consumer GPUs", section 5
// (optim="paged_adamw_32bit"), glossary "QLoRA", "How QLoRA works": the
// optimizer state lives in NVIDIA unified memory and moves to CPU RAM during
// memory spikes, so training does not fail with out-of-memory.  Only the two
// LoRA matrices are trained, so the state is small (2 x 4 B per LoRA weight).
//
// The update is AdamW with decoupled weight decay (Loshchilov and Hutter,
// "Decoupled Weight Decay Regularization", 2019), float32 state, every
// operation rounded once in float32 in this order (bit-exact against the
// definition):
//   p  = master * (1 - lr wd)
//   m  = beta1 m + (1 - beta1) g
//   v  = beta2 v + (1 - beta2) (g g)
//   p -= (lr / (1 - beta1^t)) * (m / (sqrt(v) / sqrt(1 - beta2^t) + eps))
//   master = p, param = bf16_rn(p)
// The scalar factors (1 - lr wd), 1 - beta, lr / (1 - beta1^t) and
// sqrt(1 - beta2^t) are formed on the host in double precision and rounded to
// float32.  One launch updates a whole list of tensors (the A and B of every
// adapted layer): the step is launch-bound, not bandwidth-bound.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace qlora {

constexpr int kAwMaxTensors = 240;  // per launch (kernel parameter space)
constexpr int kAwChunk = 8192;      // elements per work item
constexpr int kAwThreads = 256;

struct AwParams {
  AdamwTensor t[kAwMaxTensors];
  int64_t item0[kAwMaxTensors + 1];  // first work item of each tensor; item0[count] = total
  int count;
  float decay, beta1, omb1, beta2, omb2, step_size, bc2_sqrt, eps;
};

__device__ __forceinline__ void adamw_one(const AwParams& p, float& master, float g, float& m, float& v) {
  float w = __fmul_rn(master, p.decay);
  m = __fadd_rn(__fmul_rn(p.beta1, m), __fmul_rn(p.omb1, g));
  v = __fadd_rn(__fmul_rn(p.beta2, v), __fmul_rn(p.omb2, __fmul_rn(g, g)));
  const float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), p.bc2_sqrt), p.eps);
  w = __fsub_rn(w, __fmul_rn(p.step_size, __fdiv_rn(m, denom)));
  master = w;
}

__global__ void __launch_bounds__(kAwThreads) k_adamw(const __grid_constant__ AwParams p) {
  const int64_t total = p.item0[p.count];
  for (int64_t item = blockIdx.x; item < total; item += gridDim.x) {
    int lo = 0, hi = p.count - 1;  // tensor of this item
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.item0[mid] <= item) lo = mid; else hi = mid - 1;
    }
    const AdamwTensor& t = p.t[lo];
    const int64_t e0 = (item - p.item0[lo]) * kAwChunk;
    const int64_t e1 = min(t.numel, e0 + kAwChunk);
    for (int64_t i = e0 + threadIdx.x; i < e1; i += kAwThreads) {
      float master = t.master[i], m = t.exp_avg[i], v = t.exp_avg_sq[i];
      adamw_one(p, master, t.grad[i], m, v);
      t.master[i] = master;
      t.exp_avg[i] = m;
      t.exp_avg_sq[i] = v;
      if (t.param) t.param[i] = __float2bfloat16_rn(master);
    }
  }
}

cudaError_t launch_adamw(const AdamwTensor* tensors, int count, const AdamwHyper& h, int num_sms, cudaStream_t s) {
  for (int c0 = 0; c0 < count; c0 += kAwMaxTensors) {
    AwParams p;
    p.count = count - c0 < kAwMaxTensors ? count - c0 : kAwMaxTensors;
    int64_t items = 0;
    for (int i = 0; i < p.count; ++i) {
      p.t[i] = tensors[c0 + i];
      p.item0[i] = items;
      items += (p.t[i].numel + kAwChunk - 1) / kAwChunk;
    }
    p.item0[p.count] = items;
    p.decay = h.decay;
    p.beta1 = h.beta1;
    p.omb1 = h.omb1;
    p.beta2 = h.beta2;
    p.omb2 = h.omb2;
    p.step_size = h.step_size;
    p.bc2_sqrt = h.bc2_sqrt;
    p.eps = h.eps;
    if (items == 0) continue;
    const int64_t grid = items < 4LL * num_sms ? items : 4LL * num_sms;
    k_adamw<<<static_cast<unsigned>(grid), kAwThreads, 0, s>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

AdamwHyper adamw_hyper(double lr, double beta1, double beta2, double eps, double weight_decay, int64_t step) {
  AdamwHyper h;
  h.decay = static_cast<float>(1.0 - lr * weight_decay);
  h.beta1 = static_cast<float>(beta1);
  h.omb1 = static_cast<float>(1.0 - beta1);
  h.beta2 = static_cast<float>(beta2);
  h.omb2 = static_cast<float>(1.0 - beta2);
  h.step_size = static_cast<float>(lr / (1.0 - std::pow(beta1, static_cast<double>(step))));
  h.bc2_sqrt = static_cast<float>(std::sqrt(1.0 - std::pow(beta2, static_cast<double>(step))));
  h.eps = static_cast<float>(eps);
  return h;
}

}  // namespace qlora
