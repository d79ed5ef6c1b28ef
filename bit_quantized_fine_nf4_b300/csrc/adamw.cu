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
  griddep_wait();  // launched early: the gradients come from the preceding kernels
  griddep_launch_dependents();
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
    float* __restrict__ mp = t.master;
    const float* __restrict__ gp = t.grad;
    float* __restrict__ ap = t.exp_avg;
    float* __restrict__ vp = t.exp_avg_sq;
    __nv_bfloat16* __restrict__ pp = t.param;
    const bool vec = ((reinterpret_cast<uintptr_t>(mp) | reinterpret_cast<uintptr_t>(gp) |
                       reinterpret_cast<uintptr_t>(ap) | reinterpret_cast<uintptr_t>(vp)) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(pp) & 7u) == 0;
    int64_t i = e0 + threadIdx.x;
    if (vec) {
      // 16-byte accesses, two float4 groups per thread in flight: every load of the pair is
      // issued before the first store (e0 is a multiple of 8192, so the groups stay aligned)
      constexpr int64_t kStride = 4 * kAwThreads;
      int64_t j = e0 + 4 * threadIdx.x;
      for (; j + kStride + 4 <= e1; j += 2 * kStride) {
        float4 w[2], g[2], m[2], v[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int64_t o = j + u * kStride;
          w[u] = *reinterpret_cast<const float4*>(mp + o);
          g[u] = *reinterpret_cast<const float4*>(gp + o);
          m[u] = *reinterpret_cast<const float4*>(ap + o);
          v[u] = *reinterpret_cast<const float4*>(vp + o);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int64_t o = j + u * kStride;
          adamw_one(p, w[u].x, g[u].x, m[u].x, v[u].x);
          adamw_one(p, w[u].y, g[u].y, m[u].y, v[u].y);
          adamw_one(p, w[u].z, g[u].z, m[u].z, v[u].z);
          adamw_one(p, w[u].w, g[u].w, m[u].w, v[u].w);
          *reinterpret_cast<float4*>(mp + o) = w[u];
          *reinterpret_cast<float4*>(ap + o) = m[u];
          *reinterpret_cast<float4*>(vp + o) = v[u];
          if (pp)
            *reinterpret_cast<uint2*>(pp + o) = make_uint2(pack_bf16x2_rn(w[u].x, w[u].y), pack_bf16x2_rn(w[u].z, w[u].w));
        }
      }
      for (; j + 4 <= e1; j += kStride) {
        float4 w = *reinterpret_cast<const float4*>(mp + j), g = *reinterpret_cast<const float4*>(gp + j);
        float4 m = *reinterpret_cast<const float4*>(ap + j), v = *reinterpret_cast<const float4*>(vp + j);
        adamw_one(p, w.x, g.x, m.x, v.x);
        adamw_one(p, w.y, g.y, m.y, v.y);
        adamw_one(p, w.z, g.z, m.z, v.z);
        adamw_one(p, w.w, g.w, m.w, v.w);
        *reinterpret_cast<float4*>(mp + j) = w;
        *reinterpret_cast<float4*>(ap + j) = m;
        *reinterpret_cast<float4*>(vp + j) = v;
        if (pp) *reinterpret_cast<uint2*>(pp + j) = make_uint2(pack_bf16x2_rn(w.x, w.y), pack_bf16x2_rn(w.z, w.w));
      }
      i = e0 + ((e1 - e0) & ~int64_t(3)) + threadIdx.x;  // the last numel % 4 elements
    }
    for (; i < e1; i += kAwThreads) {
      float master = mp[i], m = ap[i], v = vp[i];
      adamw_one(p, master, gp[i], m, v);
      mp[i] = master;
      ap[i] = m;
      vp[i] = v;
      if (pp) pp[i] = __float2bfloat16_rn(master);
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
    cudaError_t e = launch_pdl_plain(k_adamw, dim3(static_cast<unsigned>(grid)), dim3(kAwThreads), 0, s, p);
    if (e == cudaSuccess) e = cudaGetLastError();
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
