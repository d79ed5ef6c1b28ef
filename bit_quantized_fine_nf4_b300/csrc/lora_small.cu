// Skinny LoRA contractions and elementwise glue.
//
// Day 25 notes "Fine-tuning and LoRA/QLoRA", section 2.1: the LoRA branch of a
// frozen linear is B (A x) with A in R^{r x k}, B in R^{d x r}; section 6.2:
// it is scaled by s = alpha / r.
//
// k_lora_down:   out[m, j] = sum_k in[m, k] * mt[j, k]   (in [M, K], mt [r, K], bf16, K % 8 == 0)
//   forward:  T = X A^T   (mt = A)
//   backward: U = dY B    (mt = B^T, made by k_transpose_bf16)
// The contraction is HBM-bound (one read of `in`, r <= 128 outputs per row),
// so it runs on the warp-level mma.sync path with 16-byte loads; the K range
// is split over the 8 warps of a CTA and over CTAs, and the partial sums are
// added in a fixed order (deterministic).
//
// The SiLU * up glue between the MLP linears is not on the pages; it is the
// plain definition h = silu(g) * u, evaluated in float32.
#include "common.cuh"
#include "kernels.h"

namespace qlora {

__device__ __forceinline__ void mma_m16n8k16_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                  uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// CTA = 8 warps, 16 rows of `in`.  Warp w handles 32-wide k chunks c with
// c % (8 * splits) == 8 * blockIdx.y + w.  Within a chunk, thread (g, q) =
// (lane / 4, lane % 4) loads 8 consecutive k (16 bytes) of rows g and g + 8,
// and the k order inside the two m16n8k16 steps is permuted consistently for
// both operands so each fragment register is one aligned 32-bit word.
template <int NT>  // number of 8-wide output column tiles (r_pad = 8 * NT)
__global__ void __launch_bounds__(256) k_lora_down(const __nv_bfloat16* __restrict__ in,
                                                   const __nv_bfloat16* __restrict__ mt, int M, int K, int r,
                                                   int splits, float* __restrict__ partial,
                                                   unsigned* __restrict__ counters, float scale,
                                                   float* __restrict__ out_f32, __nv_bfloat16* __restrict__ out_bf16) {
  constexpr int RP = NT * 8;
  extern __shared__ float s_red[];  // [8 warps][16 rows][RP]
  __shared__ int s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int m0 = blockIdx.x * 16;
  const int rowa = m0 + g, rowb = m0 + g + 8;
  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

  // K % 8 == 0: each thread's 8-element slice is either fully inside K or fully past it
  const int n_chunks = (K + 31) / 32;
  const int stride = 8 * splits;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  for (int c = 8 * blockIdx.y + warp; c < n_chunks; c += stride) {
    const int kb = c * 32 + q * 8;
    const bool kin = kb < K;
    const uint4 xa = (kin && rowa < M) ? ldg_nc_v4(in + static_cast<int64_t>(rowa) * K + kb) : zero;
    const uint4 xb = (kin && rowb < M) ? ldg_nc_v4(in + static_cast<int64_t>(rowb) * K + kb) : zero;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int j = t * 8 + g;
      const uint4 bv = (kin && j < r) ? ldg_nc_v4(mt + static_cast<int64_t>(j) * K + kb) : zero;
      mma_m16n8k16_bf16(acc[t], xa.x, xb.x, xa.y, xb.y, bv.x, bv.y);
      mma_m16n8k16_bf16(acc[t], xa.z, xb.z, xa.w, xb.w, bv.z, bv.w);
    }
  }
  // intra-CTA reduction over the 8 warps in warp order
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int col = t * 8 + 2 * q;
    float* base = s_red + warp * 16 * RP;
    base[g * RP + col] = acc[t][0];
    base[g * RP + col + 1] = acc[t][1];
    base[(g + 8) * RP + col] = acc[t][2];
    base[(g + 8) * RP + col + 1] = acc[t][3];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < 16 * RP; idx += 256) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) v += s_red[w * 16 * RP + idx];
    s_red[idx] = v;  // warp 0's slot now holds the CTA sum (each idx read before written by this thread only)
  }
  if (splits == 1) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < 16 * RP; idx += 256) {
      const int row = m0 + idx / RP, j = idx % RP;
      if (row >= M || j >= r) continue;
      const float v = s_red[idx];
      if (out_f32) out_f32[static_cast<int64_t>(row) * r + j] = v;
      if (out_bf16) out_bf16[static_cast<int64_t>(row) * r + j] = __float2bfloat16_rn(__fmul_rn(v, scale));
    }
    return;
  }
  // split-K over CTAs: publish, last CTA of this row tile adds the splits in order
  float* mine = partial + (static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x) * 16 * RP;
  __syncthreads();
  for (int idx = threadIdx.x; idx < 16 * RP; idx += 256) mine[idx] = s_red[idx];
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(counters + blockIdx.x, 1u) == static_cast<unsigned>(splits - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int idx = threadIdx.x; idx < 16 * RP; idx += 256) {
    float v = 0.f;
    for (int sp = 0; sp < splits; ++sp)
      v += __ldcg(partial + (static_cast<int64_t>(sp) * gridDim.x + blockIdx.x) * 16 * RP + idx);
    const int row = m0 + idx / RP, j = idx % RP;
    if (row >= M || j >= r) continue;
    if (out_f32) out_f32[static_cast<int64_t>(row) * r + j] = v;
    if (out_bf16) out_bf16[static_cast<int64_t>(row) * r + j] = __float2bfloat16_rn(__fmul_rn(v, scale));
  }
  if (threadIdx.x == 0) counters[blockIdx.x] = 0;
}

// dst[c, r] = src[r, c]   (bf16, rows x cols source)
__global__ void k_transpose_bf16(const __nv_bfloat16* __restrict__ src, __nv_bfloat16* __restrict__ dst, int rows,
                                 int cols) {
  __shared__ __nv_bfloat16 tile[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int rr = r0 + i, cc = c0 + threadIdx.x;
    if (rr < rows && cc < cols) tile[i][threadIdx.x] = src[static_cast<int64_t>(rr) * cols + cc];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int cc = c0 + i, rr = r0 + threadIdx.x;
    if (rr < rows && cc < cols) dst[static_cast<int64_t>(cc) * rows + rr] = tile[threadIdx.x][i];
  }
}

// dst = bf16_rn(scale * src)
__global__ void k_scale_to_bf16(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst, int64_t n,
                                float scale) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    dst[i] = __float2bfloat16_rn(__fmul_rn(src[i], scale));
}

// ------------------------------------------------------------------ SiLU * up
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float sigmoidf_(float g) { return 1.0f / (1.0f + expf(-g)); }

__global__ void __launch_bounds__(256) k_silu_mul_fwd(const uint32_t* __restrict__ g, const uint32_t* __restrict__ u,
                                                      uint32_t* __restrict__ h, int64_t n2) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n2;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint32_t gw = g[i], uw = u[i];
    float o[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const float gv = t ? bf_hi(gw) : bf_lo(gw), uv = t ? bf_hi(uw) : bf_lo(uw);
      o[t] = gv * sigmoidf_(gv) * uv;
    }
    h[i] = pack_bf16x2_rn(o[0], o[1]);
  }
}

__global__ void __launch_bounds__(256) k_silu_mul_bwd(const uint32_t* __restrict__ dh, const uint32_t* __restrict__ g,
                                                      const uint32_t* __restrict__ u, uint32_t* __restrict__ dg,
                                                      uint32_t* __restrict__ du, int64_t n2) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n2;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint32_t dw = dh[i], gw = g[i], uw = u[i];
    float og[2], ou[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const float d = t ? bf_hi(dw) : bf_lo(dw), gv = t ? bf_hi(gw) : bf_lo(gw), uv = t ? bf_hi(uw) : bf_lo(uw);
      const float sg = sigmoidf_(gv);
      ou[t] = d * gv * sg;
      og[t] = d * uv * sg * (1.0f + gv * (1.0f - sg));
    }
    dg[i] = pack_bf16x2_rn(og[0], og[1]);
    du[i] = pack_bf16x2_rn(ou[0], ou[1]);
  }
}

// ------------------------------------------------------------------ launchers
int lora_down_splits(int M, int K, int num_sms) {
  const int tiles = M > 0 ? (M + 15) / 16 : 1;
  int splits = 1;
  while (tiles * splits < num_sms && splits * 2 * 8 * 32 <= K) splits *= 2;
  return splits;
}

size_t lora_down_workspace_bytes(int M, int K, int r, int num_sms) {
  const int splits = lora_down_splits(M, K, num_sms);
  if (splits == 1) return 0;
  const int tiles = (M + 15) / 16;
  const int rp = r <= 16 ? 16 : (r <= 32 ? 32 : (r <= 64 ? 64 : 128));
  return static_cast<size_t>(splits) * tiles * 16 * rp * sizeof(float) + static_cast<size_t>(tiles) * 4 + 256;
}

cudaError_t launch_lora_down(const __nv_bfloat16* in, const __nv_bfloat16* mt, int M, int K, int r, float scale,
                             float* out_f32, __nv_bfloat16* out_bf16, void* ws, int num_sms, cudaStream_t s) {
  const int tiles = (M + 15) / 16;
  const int splits = lora_down_splits(M, K, num_sms);
  const int rp = r <= 16 ? 16 : (r <= 32 ? 32 : (r <= 64 ? 64 : 128));
  float* partial = nullptr;
  unsigned* counters = nullptr;
  if (splits > 1) {
    partial = static_cast<float*>(ws);
    counters = reinterpret_cast<unsigned*>(partial + static_cast<size_t>(splits) * tiles * 16 * rp);
    cudaError_t e = cudaMemsetAsync(counters, 0, static_cast<size_t>(tiles) * 4, s);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid(tiles, splits);
  const size_t smem = static_cast<size_t>(8) * 16 * rp * sizeof(float);
#define QLORA_LD(NT)                                                                                          \
  do {                                                                                                        \
    cudaFuncSetAttribute(k_lora_down<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)); \
    k_lora_down<NT><<<grid, 256, smem, s>>>(in, mt, M, K, r, splits, partial, counters, scale, out_f32, out_bf16); \
  } while (0)
  if (rp == 16) QLORA_LD(2);
  else if (rp == 32) QLORA_LD(4);
  else if (rp == 64) QLORA_LD(8);
  else QLORA_LD(16);
#undef QLORA_LD
  return cudaGetLastError();
}

cudaError_t launch_transpose_bf16(const __nv_bfloat16* src, __nv_bfloat16* dst, int rows, int cols, cudaStream_t s) {
  const dim3 grid((cols + 31) / 32, (rows + 31) / 32), block(32, 8);
  k_transpose_bf16<<<grid, block, 0, s>>>(src, dst, rows, cols);
  return cudaGetLastError();
}

cudaError_t launch_scale_to_bf16(const float* src, __nv_bfloat16* dst, int64_t n, float scale, int num_sms,
                                 cudaStream_t s) {
  int64_t g = (n + 255) / 256;
  if (g > num_sms * 8) g = num_sms * 8;
  if (g < 1) g = 1;
  k_scale_to_bf16<<<static_cast<unsigned>(g), 256, 0, s>>>(src, dst, n, scale);
  return cudaGetLastError();
}

cudaError_t launch_silu_mul_fwd(const uint16_t* g, const uint16_t* u, uint16_t* h, int64_t n, int num_sms,
                                cudaStream_t s) {
  const int64_t n2 = n / 2;
  int64_t grid = (n2 + 255) / 256;
  if (grid > num_sms * 16) grid = num_sms * 16;
  if (grid < 1) grid = 1;
  k_silu_mul_fwd<<<static_cast<unsigned>(grid), 256, 0, s>>>(reinterpret_cast<const uint32_t*>(g),
                                                             reinterpret_cast<const uint32_t*>(u),
                                                             reinterpret_cast<uint32_t*>(h), n2);
  return cudaGetLastError();
}

cudaError_t launch_silu_mul_bwd(const uint16_t* dh, const uint16_t* g, const uint16_t* u, uint16_t* dg, uint16_t* du,
                                int64_t n, int num_sms, cudaStream_t s) {
  const int64_t n2 = n / 2;
  int64_t grid = (n2 + 255) / 256;
  if (grid > num_sms * 16) grid = num_sms * 16;
  if (grid < 1) grid = 1;
  k_silu_mul_bwd<<<static_cast<unsigned>(grid), 256, 0, s>>>(
      reinterpret_cast<const uint32_t*>(dh), reinterpret_cast<const uint32_t*>(g),
      reinterpret_cast<const uint32_t*>(u), reinterpret_cast<uint32_t*>(dg), reinterpret_cast<uint32_t*>(du), n2);
  return cudaGetLastError();
}

}  // namespace qlora
