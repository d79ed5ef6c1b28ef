// LoRA dropout: the counter-based keep mask and its application to the branch input.
//
// Every page's LoRA configuration sets lora_dropout = 0.05 (P1 tutorial "QLoRA:
// fine-tuning 7B on a 24 GB card", section 3.3; tbr8.org "QLoRA on consumer
// GPUs", section 4; fedte.cc "QLoRA fine-tuning on 4 GB", section 2).  Dropout
// acts on the input of the LoRA branch: B A (x * m) / (1 - p), the frozen path
// sees x.
//
// Mask: Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers:
// as easy as 1, 2, 3", SC 2011).  Element e = row * k + col of the [m, k]
// input takes word e % 4 of Philox(counter = (e / 4 as two 32-bit words,
// offset as two 32-bit words), key = seed as two 32-bit words) and is kept when
// the word is >= floor(p 2^32).  One bit per element, least significant first:
// byte e / 8, bit e % 8 (a row of k % 64 == 0 elements is k / 8 whole bytes).
// One thread makes one 32-bit mask word (8 Philox calls, 32 elements).
#include "common.cuh"
#include "kernels.h"

namespace qlora {

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
  constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u, kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
#pragma unroll
  for (int rnd = 0; rnd < 10; ++rnd) {
    if (rnd > 0) {
      k0 += kW0;
      k1 += kW1;
    }
    const uint32_t hi0 = __umulhi(kM0, c.x), lo0 = kM0 * c.x;
    const uint32_t hi1 = __umulhi(kM1, c.z), lo1 = kM1 * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

__global__ void __launch_bounds__(256) k_dropout_mask(uint32_t* __restrict__ mask, int64_t n_words, uint64_t seed,
                                                      uint64_t offset, uint32_t threshold) {
  griddep_wait();  // launched early: the previous mask may still be read by the preceding kernels
  griddep_launch_dependents();
  const uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
  const uint32_t o0 = static_cast<uint32_t>(offset), o1 = static_cast<uint32_t>(offset >> 32);
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; w < n_words;
       w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    uint32_t bits = 0;
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const uint64_t grp = static_cast<uint64_t>(w) * 8 + g;  // counter of elements 4 grp .. 4 grp + 3
      const uint4 r = philox4x32_10(make_uint4(static_cast<uint32_t>(grp), static_cast<uint32_t>(grp >> 32), o0, o1),
                                    k0, k1);
      bits |= (r.x >= threshold ? 1u : 0u) << (4 * g);
      bits |= (r.y >= threshold ? 1u : 0u) << (4 * g + 1);
      bits |= (r.z >= threshold ? 1u : 0u) << (4 * g + 2);
      bits |= (r.w >= threshold ? 1u : 0u) << (4 * g + 3);
    }
    mask[w] = bits;
  }
}

// x_drop[e] = keep(e) ? x[e] : 0 (bf16, exact); 8 elements (one mask byte) per thread step.
__global__ void __launch_bounds__(256) k_dropout_apply(const uint4* __restrict__ x, const uint8_t* __restrict__ mask,
                                                       uint4* __restrict__ x_drop, int64_t n8) {
  griddep_wait();  // launched early: x and the mask come from the preceding kernels
  griddep_launch_dependents();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 v = x[i];
    const uint32_t b = mask[i];
    auto sel = [&](uint32_t word, int t) {  // keep the bf16 halves whose bits (t, t + 1) are set
      const uint32_t lo = (b >> t) & 1u ? 0x0000ffffu : 0u;
      const uint32_t hi = (b >> (t + 1)) & 1u ? 0xffff0000u : 0u;
      return word & (lo | hi);
    };
    x_drop[i] = make_uint4(sel(v.x, 0), sel(v.y, 2), sel(v.z, 4), sel(v.w, 6));
  }
}

uint32_t dropout_threshold(float p) {
  const double t = static_cast<double>(p) * 4294967296.0;
  return static_cast<uint32_t>(t);  // floor for 0 <= p < 1
}

cudaError_t launch_dropout_mask(uint64_t seed, uint64_t offset, int64_t n_elems, float p, uint8_t* mask, int num_sms,
                                cudaStream_t s) {
  const int64_t n_words = n_elems / 32;  // n_elems is a multiple of 64
  if (n_words == 0) return cudaSuccess;
  int64_t grid = (n_words + 255) / 256;
  if (grid > 8LL * num_sms) grid = 8LL * num_sms;
  const cudaError_t e = launch_pdl_plain(k_dropout_mask, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s,
                                         reinterpret_cast<uint32_t*>(mask), n_words, seed, offset, dropout_threshold(p));
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_dropout_apply(const uint16_t* x, const uint8_t* mask, uint16_t* x_drop, int64_t n_elems, int num_sms,
                                 cudaStream_t s) {
  const int64_t n8 = n_elems / 8;
  if (n8 == 0) return cudaSuccess;
  int64_t grid = (n8 + 255) / 256;
  if (grid > 16LL * num_sms) grid = 16LL * num_sms;
  const cudaError_t e = launch_pdl_plain(k_dropout_apply, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s,
                                         reinterpret_cast<const uint4*>(x), mask, reinterpret_cast<uint4*>(x_drop), n8);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qlora
