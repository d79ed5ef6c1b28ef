// Skinny LoRA contractions and elementwise glue.
//
// Day 25 notes "Fine-tuning and LoRA/QLoRA", section 2.1: the LoRA branch of a
// frozen linear is B (A x) with A in R^{r x k}, B in R^{d x r}; section 6.2:
// it is scaled by s = alpha / r.
//
// k_lora_down:   out[m, j] = sum_k in[m, k] * mt(j, k)   (in [M, K] bf16, K % 8 == 0)
//   forward:  T = X A^T   (mt = A, [r, K])
//   backward: U = dY B    (mt = B as stored, [N, r])
// The contraction is HBM-bound (one read of `in`, r <= 128 outputs per row),
// so it runs on the warp-level mma.sync path with 16-byte loads.  The grid is
// persistent and capped by the caller (it runs on the SMs a GEMM leaves idle);
// the K range of a 16-row tile is split over the warps of one CTA and the
// partial sums are added in warp order (deterministic, no cross-CTA step).
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

// Persistent CTAs of W warps walk 16-row tiles of `in` (tile = blockIdx.x,
// += gridDim.x); the W warps of a CTA split k (32-wide chunks, chunk c taken by
// warp c % W, 4 or 2 chunks per loop trip so their loads are in flight
// together) and add their partial sums in warp order.  Within a chunk, thread
// (g, q) = (lane / 4, lane % 4) loads 8 consecutive k (16 bytes) of rows g and
// g + 8, and the k order inside the two m16n8k16 steps is permuted the same way
// for both operands so each fragment register holds 2 consecutive k.
// MT_KMAJOR: mt is [r, K] (row j contiguous in k); otherwise mt is [K, r]
// (the LoRA B matrix as stored).  STAGED: the CTA first copies mt into shared
// memory as [RP rows j][K] (transposing [K, r]), rows padded by 16 bytes so the
// 16-byte fragment loads of 8 rows x 4 threads hit distinct bank groups; every
// tile then reads its fragments from there.  Unstaged, fragments come from
// global memory (and gather 8 strided values when mt is [K, r]).
// Outputs (out = t_scale * in . mt^T, t_scale = 1 except under dropout):
// out_f32 [M, r] (row stride r) and out_bf16 = bf16(scale * out)
// [M, rk] with rk = r rounded up to a multiple of 8 (the row stride of the
// internal bf16 LoRA operands, which the tensor-core kernels load by TMA); its
// columns r .. rk-1 are zero.
// Side job (optional): cvt_dst[i, j] = bf16(cvt_scale * cvt_src[i, j]) for the
// cvt_rows x r matrix cvt_src (row stride r) into cvt_dst (row stride rk, zero
// in columns r .. rk-1), spread over all threads of the grid -- an independent
// elementwise pass in the same launch.
template <int NT, bool MT_KMAJOR>
__device__ __forceinline__ uint4 load_mt_frag(const __nv_bfloat16* __restrict__ mt, int j, int kb, int K, int r) {
  if (MT_KMAJOR) return ldg_nc_v4(mt + static_cast<int64_t>(j) * K + kb);
  const unsigned short* p = reinterpret_cast<const unsigned short*>(mt) + static_cast<int64_t>(kb) * r + j;
  uint32_t v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __ldg(p + static_cast<int64_t>(i) * r);
  return make_uint4(v[0] | (v[1] << 16), v[2] | (v[3] << 16), v[4] | (v[5] << 16), v[6] | (v[7] << 16));
}

template <int NT, bool MT_KMAJOR, int W, bool STAGED>
__global__ void __launch_bounds__(W * 32) k_lora_down(const __nv_bfloat16* __restrict__ in,
                                                      const __nv_bfloat16* __restrict__ mt, int M, int K, int r,
                                                      float scale, float* __restrict__ out_f32,
                                                      __nv_bfloat16* __restrict__ out_bf16,
                                                      const float* __restrict__ cvt_src,
                                                      __nv_bfloat16* __restrict__ cvt_dst, int64_t cvt_rows,
                                                      float cvt_scale, float t_scale) {
  constexpr int RP = NT * 8;
  extern __shared__ float s_red[];  // [W warps][16 rows][RP], then (STAGED) mt as [RP][K + 8] bf16
  unsigned short* s_mt = reinterpret_cast<unsigned short*>(s_red + W * 16 * RP);
  const int mt_pitch = K + 8;
  // launched early (programmatic dependent launch): `in`, the LoRA matrix (an optimiser step may
  // have just written it), t_save and the outputs may belong to the preceding kernels of the stream
  griddep_wait();
  // the GEMM that consumes this kernel's output only needs it for its last k block; it may start
  // now, since every kernel before this one has completed
  griddep_launch_dependents();
  if (STAGED) {
    if (MT_KMAJOR) {
      // rows j < r: 16-byte copies; rows r .. RP - 1: zero
      const int per_row = K / 8;
      for (int i = threadIdx.x; i < RP * per_row; i += W * 32) {
        const int j = i / per_row, c = (i - j * per_row) * 8;
        const uint4 v = j < r ? ldg_nc_v4(mt + static_cast<int64_t>(j) * K + c) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(s_mt + j * mt_pitch + c) = v;
      }
    } else {
      // mt[k][j] -> s_mt[j][k]; one thread per (k, 8 j)
      const int jg = RP / 8;
      const int total = K * jg;
      if ((r & 7) == 0) {
        // rows of mt start on 16-byte boundaries: 16-byte loads, eight in flight per thread
        for (int i0 = threadIdx.x; i0 < total; i0 += 8 * W * 32) {
          uint4 v[8];
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            const int i = i0 + b * W * 32;
            const int k = i / jg, j0 = (i - k * jg) * 8;
            v[b] = (i < total && j0 < r)
                       ? ldg_nc_v4(reinterpret_cast<const unsigned short*>(mt) + static_cast<int64_t>(k) * r + j0)
                       : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            const int i = i0 + b * W * 32;
            if (i >= total) break;
            const int k = i / jg, j0 = (i - k * jg) * 8;
            const uint32_t w[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              s_mt[(j0 + 2 * e) * mt_pitch + k] = static_cast<unsigned short>(w[e] & 0xffffu);
              s_mt[(j0 + 2 * e + 1) * mt_pitch + k] = static_cast<unsigned short>(w[e] >> 16);
            }
          }
        }
      } else {
        for (int i = threadIdx.x; i < total; i += W * 32) {
          const int k = i / jg, j0 = (i - k * jg) * 8;
          const unsigned short* src = reinterpret_cast<const unsigned short*>(mt) + static_cast<int64_t>(k) * r;
#pragma unroll
          for (int e = 0; e < 8; ++e) s_mt[(j0 + e) * mt_pitch + k] = j0 + e < r ? src[j0 + e] : 0;
        }
      }
    }
    __syncthreads();
  }
  const int rk = (r + 7) & ~7;
  if (cvt_rows > 0) {
    const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t n_out = cvt_rows * rk;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_out; i += nthreads) {
      const int64_t row = i / rk;
      const int j = static_cast<int>(i - row * rk);
      cvt_dst[i] = j < r ? __float2bfloat16_rn(__fmul_rn(cvt_src[row * r + j], cvt_scale)) : __float2bfloat16_rn(0.f);
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int n_chunks = (K + 31) / 32;  // K % 8 == 0: a thread's 8-wide slice is fully inside K or past it
  const int tiles = (M + 15) / 16;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  // staged: the LoRA fragments come from shared memory as the MMAs need them, so eight chunks of
  // `in` (128 KB per CTA) can be in flight; unstaged: fragments are loaded with the chunk
  constexpr int UNROLL = (NT <= 2 && STAGED) ? 8 : (NT <= 2 && MT_KMAJOR) ? 4 : 2;
  constexpr int BV = STAGED ? 1 : UNROLL;
  for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int m0 = tile * 16;
    const int rowa = m0 + g, rowb = m0 + g + 8;
    const __nv_bfloat16* ina = in + static_cast<int64_t>(rowa) * K;
    const __nv_bfloat16* inb = in + static_cast<int64_t>(rowb) * K;
    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
    for (int c = warp; c < n_chunks; c += UNROLL * W) {
      uint4 xa[UNROLL], xb[UNROLL], bv[BV][NT];
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const int kb = (c + u * W) * 32 + q * 8;
        const bool kin = kb < K;
        xa[u] = (kin && rowa < M) ? ldg_nc_v4(ina + kb) : zero;
        xb[u] = (kin && rowb < M) ? ldg_nc_v4(inb + kb) : zero;
        if (!STAGED) {
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const int j = t * 8 + g;
            bv[u % BV][t] = (kin && j < r) ? load_mt_frag<NT, MT_KMAJOR>(mt, j, kb, K, r) : zero;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        if (STAGED) {
          const int kb = (c + u * W) * 32 + q * 8;
#pragma unroll
          for (int t = 0; t < NT; ++t)
            bv[0][t] = kb < K ? *reinterpret_cast<const uint4*>(s_mt + (t * 8 + g) * mt_pitch + kb) : zero;
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const uint4 bw = bv[u % BV][t];
          mma_m16n8k16_bf16(acc[t], xa[u].x, xb[u].x, xa[u].y, xb[u].y, bw.x, bw.y);
          mma_m16n8k16_bf16(acc[t], xa[u].z, xb[u].z, xa[u].w, xb[u].w, bw.z, bw.w);
        }
      }
    }
    // reduction over the W warps in warp order
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
    for (int idx = threadIdx.x; idx < 16 * RP; idx += W * 32) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < W; ++w) v += s_red[w * 16 * RP + idx];
      v = __fmul_rn(v, t_scale);  // 1 except under dropout (1 / (1 - p))
      const int row = m0 + idx / RP, j = idx % RP;
      if (row >= M) continue;
      // columns j >= r of the product are exactly zero (mt rows past r load as zero)
      if (out_f32 && j < r) out_f32[static_cast<int64_t>(row) * r + j] = v;
      if (out_bf16 && j < rk) out_bf16[static_cast<int64_t>(row) * rk + j] = __float2bfloat16_rn(__fmul_rn(v, scale));
    }
    __syncthreads();  // s_red is reused by the next tile
  }
}

// ------------------------------------------------------------------ U = dY B, k split over a cluster
// The backward's U for r <= 16 when the tokens fill no more than a wave of 64-row blocks: a CTA
// takes 64 rows and a 1/S share of k (the S shares of a row block form one cluster, S <= 4).  It
// stages only its k slice of mt, transposed to [RP rows j][slice] bf16 (row pitch = 64 bytes past
// a multiple of 128, so the 16-byte fragment loads of a quarter warp hit distinct bank groups),
// and its 16 warps (row group = warp % 4, k part = warp / 4, 32-wide chunks taken in turn) issue
// all 16-byte loads of up to 8 chunks before the first MMA: 8 KB per warp, 128 KB per CTA in
// flight (the first such trip before the slice of mt is staged, so the two overlap).  Sums, all in
// a fixed order: the four k parts of a row group in shared memory, then the
// S ranks' partials sent with st.shared::cluster to the rank owning the row group (group % S) and
// added there in rank order.  Outputs and the side job as in k_lora_down.
constexpr int kLdkThreads = 512;
constexpr int kLdkGroups = 4;                      // 16-row groups per CTA
constexpr int kLdkRows = 16 * kLdkGroups;          // rows per CTA
constexpr int kLdkParts = 16 / kLdkGroups;         // warps along k per row group
constexpr int kLdkMaxSplits = 4;                   // cluster size
constexpr int kLdkUnroll = 8;                      // chunks in flight per warp
constexpr size_t kLdkMaxSliceBytes = 160 * 1024;   // staged mt slice per CTA

__host__ __device__ inline int ldk_pitch(int chunks_per_split) {
  return ((chunks_per_split * 32 + 63) & ~63) + 32;  // bf16 elements
}
__host__ __device__ inline size_t ldk_smem_bytes(int rp, int chunks_per_split, int splits) {
  const int owned = (kLdkGroups + splits - 1) / splits;
  return static_cast<size_t>(rp) * ldk_pitch(chunks_per_split) * 2 +                    // mt slice
         static_cast<size_t>(kLdkGroups) * (kLdkParts - 1) * 16 * rp * sizeof(float) +  // k parts 1..3
         static_cast<size_t>(splits) * owned * 16 * rp * sizeof(float);                  // cluster slots
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
__device__ __forceinline__ void st_cluster_v2(uint32_t local, uint32_t rank, float a, float b) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local), "r"(rank));
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(ra), "f"(a), "f"(b) : "memory");
}

template <int NT, bool MT_KMAJOR>
__global__ void __launch_bounds__(kLdkThreads, 1) k_lora_down_ks(const __nv_bfloat16* __restrict__ in,
                                                                 const __nv_bfloat16* __restrict__ mt, int M, int K,
                                                                 int r, int chunks_per_split, float scale,
                                                                 float* __restrict__ out_f32,
                                                                 __nv_bfloat16* __restrict__ out_bf16,
                                                                 const float* __restrict__ cvt_src,
                                                                 __nv_bfloat16* __restrict__ cvt_dst, int64_t cvt_rows,
                                                                 float cvt_scale, float t_scale) {
  constexpr int RP = NT * 8;
  extern __shared__ __align__(16) unsigned char ldk_smem[];
  const int S = static_cast<int>(gridDim.x);  // the cluster: the k shares of one row block
  const int split = static_cast<int>(blockIdx.x);
  const int m0 = static_cast<int>(blockIdx.y) * kLdkRows;
  const int nc = (K + 31) / 32;
  const int c0 = split * chunks_per_split;
  const int c1 = min(nc, c0 + chunks_per_split);  // the host makes every share non-empty
  const int pitch = ldk_pitch(chunks_per_split);
  const int owned = (kLdkGroups + S - 1) / S;
  unsigned short* s_mt = reinterpret_cast<unsigned short*>(ldk_smem);                // [RP][pitch]
  float* s_part = reinterpret_cast<float*>(ldk_smem + static_cast<size_t>(RP) * pitch * 2);  // [group][part-1][16][RP]
  float* s_slot = s_part + kLdkGroups * (kLdkParts - 1) * 16 * RP;                   // [S][owned][16][RP]
  const uint4 zero = make_uint4(0, 0, 0, 0);

  cluster_arrive_relaxed();  // matched by the wait before the first store into another CTA
  // launched early (programmatic dependent launch): `in`, the LoRA matrix, t_save and the outputs
  // may belong to the preceding kernels of the stream
  griddep_wait();
  // the GEMM that consumes U only needs it for its last k block
  griddep_launch_dependents();

  // ---- the first trip's loads of `in`, issued before mt is staged so the two overlap
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int grp = warp % kLdkGroups, part = warp / kLdkGroups;
  const int rowa = m0 + grp * 16 + g, rowb = rowa + 8;
  const __nv_bfloat16* ina = in + static_cast<int64_t>(rowa) * K;
  const __nv_bfloat16* inb = in + static_cast<int64_t>(rowb) * K;
  uint4 xa[kLdkUnroll], xb[kLdkUnroll];
  auto load_trip = [&](int c) {
#pragma unroll
    for (int u = 0; u < kLdkUnroll; ++u) {
      const int cc = c + u * kLdkParts;
      const int kb = cc * 32 + q * 8;
      const bool kin = cc < c1 && kb < K;
      xa[u] = (kin && rowa < M) ? ldg_nc_v4(ina + kb) : zero;
      xb[u] = (kin && rowb < M) ? ldg_nc_v4(inb + kb) : zero;
    }
  };
  const int c_first = c0 + part;
  load_trip(c_first);

  // ---- stage mt[k0, k0 + 32 (c1 - c0)) as s_mt[j][k - k0] (zero for j >= r and k >= K)
  const int k0 = c0 * 32;
  const int klen = (c1 - c0) * 32;
  if (MT_KMAJOR) {
    const int per_row = klen / 8;
    for (int i = threadIdx.x; i < RP * per_row; i += kLdkThreads) {
      const int j = i / per_row, c = (i - j * per_row) * 8;
      const int k = k0 + c;  // K % 8 == 0: the 8 values lie wholly inside or wholly past K
      const uint4 v = (j < r && k < K) ? ldg_nc_v4(mt + static_cast<int64_t>(j) * K + k) : zero;
      *reinterpret_cast<uint4*>(s_mt + j * pitch + c) = v;
    }
  } else if ((r & 7) == 0) {
    // rows of mt start on 16-byte boundaries: one 16-byte load per (k, 8 j), four in flight per thread
    constexpr int JG = RP / 8;
    const int total = klen * JG;
    for (int i0 = threadIdx.x; i0 < total; i0 += 4 * kLdkThreads) {
      uint4 v[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int i = i0 + b * kLdkThreads;
        const int kk = i / JG, j0 = (i - kk * JG) * 8;
        const int k = k0 + kk;
        v[b] = (i < total && k < K && j0 < r)
                   ? ldg_nc_v4(reinterpret_cast<const unsigned short*>(mt) + static_cast<int64_t>(k) * r + j0)
                   : zero;
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int i = i0 + b * kLdkThreads;
        if (i >= total) break;
        const int kk = i / JG, j0 = (i - kk * JG) * 8;
        const uint32_t w[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          s_mt[(j0 + 2 * e) * pitch + kk] = static_cast<unsigned short>(w[e] & 0xffffu);
          s_mt[(j0 + 2 * e + 1) * pitch + kk] = static_cast<unsigned short>(w[e] >> 16);
        }
      }
    }
  } else {
    constexpr int JG = RP / 8;
    for (int i = threadIdx.x; i < klen * JG; i += kLdkThreads) {
      const int kk = i / JG, j0 = (i - kk * JG) * 8;
      const int k = k0 + kk;
      const unsigned short* src = reinterpret_cast<const unsigned short*>(mt) + static_cast<int64_t>(k) * r;
#pragma unroll
      for (int e = 0; e < 8; ++e) s_mt[(j0 + e) * pitch + kk] = (k < K && j0 + e < r) ? src[j0 + e] : 0;
    }
  }
  // ---- side job: cvt_dst = bf16(cvt_scale * cvt_src), over every thread of the grid
  const int rk = (r + 7) & ~7;
  if (cvt_rows > 0) {
    const int64_t nthreads = static_cast<int64_t>(gridDim.x) * gridDim.y * blockDim.x;
    const int64_t n_out = cvt_rows * rk;
    const int64_t b = static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x;
    for (int64_t i = b * blockDim.x + threadIdx.x; i < n_out; i += nthreads) {
      const int64_t row = i / rk;
      const int j = static_cast<int>(i - row * rk);
      cvt_dst[i] = j < r ? __float2bfloat16_rn(__fmul_rn(cvt_src[row * r + j], cvt_scale)) : __float2bfloat16_rn(0.f);
    }
  }
  __syncthreads();

  // ---- the k loop: every load of a trip issued before its MMAs
  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  for (int c = c_first; c < c1; c += kLdkParts * kLdkUnroll) {
    if (c != c_first) load_trip(c);
#pragma unroll
    for (int u = 0; u < kLdkUnroll; ++u) {
      const int cc = c + u * kLdkParts;
      if (cc >= c1) break;  // warp-uniform
      const int kl = (cc - c0) * 32 + q * 8;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const uint4 bv = *reinterpret_cast<const uint4*>(s_mt + (t * 8 + g) * pitch + kl);
        mma_m16n8k16_bf16(acc[t], xa[u].x, xb[u].x, xa[u].y, xb[u].y, bv.x, bv.y);
        mma_m16n8k16_bf16(acc[t], xa[u].z, xb[u].z, xa[u].w, xb[u].w, bv.z, bv.w);
      }
    }
  }

  // ---- the k parts of a row group, added in part order by part 0
  if (part > 0) {
    float* dst = s_part + ((grp * (kLdkParts - 1) + part - 1) * 16) * RP;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int col = t * 8 + 2 * q;
      *reinterpret_cast<float2*>(dst + g * RP + col) = make_float2(acc[t][0], acc[t][1]);
      *reinterpret_cast<float2*>(dst + (g + 8) * RP + col) = make_float2(acc[t][2], acc[t][3]);
    }
  }
  __syncthreads();
  cluster_wait();  // every CTA of the cluster has started: its shared memory may be written
  if (part == 0) {
#pragma unroll
    for (int pp = 0; pp < kLdkParts - 1; ++pp) {
      const float* src = s_part + ((grp * (kLdkParts - 1) + pp) * 16) * RP;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int col = t * 8 + 2 * q;
        const float2 a = *reinterpret_cast<const float2*>(src + g * RP + col);
        const float2 b = *reinterpret_cast<const float2*>(src + (g + 8) * RP + col);
        acc[t][0] += a.x;
        acc[t][1] += a.y;
        acc[t][2] += b.x;
        acc[t][3] += b.y;
      }
    }
    // to the owner of this row group: slot [split][grp / S]
    const uint32_t owner = static_cast<uint32_t>(grp % S);
    const uint32_t dst = smem_u32(s_slot + ((split * owned + grp / S) * 16) * RP);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int col = t * 8 + 2 * q;
      st_cluster_v2(dst + static_cast<uint32_t>((g * RP + col) * 4), owner, acc[t][0], acc[t][1]);
      st_cluster_v2(dst + static_cast<uint32_t>(((g + 8) * RP + col) * 4), owner, acc[t][2], acc[t][3]);
    }
  }
  cluster_sync();  // the slots have landed

  // ---- the owner adds the S shares in rank order and writes its row groups
  for (int idx = threadIdx.x; idx < owned * 16 * RP; idx += kLdkThreads) {
    const int gi = idx / (16 * RP), rem = idx - gi * 16 * RP;
    const int grp_o = gi * S + split;
    if (grp_o >= kLdkGroups) continue;
    float v = 0.f;
    for (int s = 0; s < S; ++s) v += s_slot[((s * owned + gi) * 16) * RP + rem];
    v = __fmul_rn(v, t_scale);
    const int row = m0 + grp_o * 16 + rem / RP, j = rem % RP;
    if (row >= M) continue;
    // columns j >= r of the product are exactly zero (mt rows past r are staged as zero)
    if (out_f32 && j < r) out_f32[static_cast<int64_t>(row) * r + j] = v;
    if (out_bf16 && j < rk) out_bf16[static_cast<int64_t>(row) * rk + j] = __float2bfloat16_rn(__fmul_rn(v, scale));
  }
}

// ------------------------------------------------------------------ SiLU * up
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float sigmoidf_(float g) { return 1.0f / (1.0f + expf(-g)); }

__global__ void __launch_bounds__(256) k_silu_mul_fwd(const uint32_t* __restrict__ g, const uint32_t* __restrict__ u,
                                                      uint32_t* __restrict__ h, int64_t n2) {
  griddep_wait();  // launched early: g and u come from the preceding kernels
  griddep_launch_dependents();
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
  griddep_wait();  // launched early: dh comes from the preceding kernels
  griddep_launch_dependents();
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
size_t lora_down_workspace_bytes(int M, int K, int r, int num_sms) {
  (void)M, (void)K, (void)r, (void)num_sms;
  return 0;  // no cross-CTA reduction
}

// mtk[j, k] = mt[k, j]: one thread per (8 consecutive k, j), j fastest so a warp reads whole rows
// of mt.  Side jobs in the same launch: cvt_dst = bf16(cvt_scale * cvt_src) as in k_lora_down, and
// zero_words words of `zero` cleared.
__global__ void __launch_bounds__(256) k_transpose_kr(const unsigned short* __restrict__ mt,
                                                      unsigned short* __restrict__ mtk, int K, int r,
                                                      const float* __restrict__ cvt_src,
                                                      __nv_bfloat16* __restrict__ cvt_dst, int64_t cvt_rows,
                                                      float cvt_scale, unsigned* __restrict__ zero, int zero_words) {
  griddep_wait();  // launched early: the workspace it writes may be in use by the preceding kernels
  griddep_launch_dependents();
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < zero_words; i += nthreads) zero[i] = 0u;
  const int64_t total = static_cast<int64_t>(K / 8) * r;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += nthreads) {
    const int j = static_cast<int>(i % r);
    const int64_t k0 = (i / r) * 8;
    uint32_t v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = __ldg(mt + (k0 + e) * r + j);
    *reinterpret_cast<uint4*>(mtk + static_cast<int64_t>(j) * K + k0) =
        make_uint4(v[0] | (v[1] << 16), v[2] | (v[3] << 16), v[4] | (v[5] << 16), v[6] | (v[7] << 16));
  }
  const int rk = (r + 7) & ~7;
  const int64_t n_out = cvt_rows * rk;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_out; i += nthreads) {
    const int64_t row = i / rk;
    const int j = static_cast<int>(i - row * rk);
    cvt_dst[i] = j < r ? __float2bfloat16_rn(__fmul_rn(cvt_src[row * r + j], cvt_scale)) : __float2bfloat16_rn(0.f);
  }
}

cudaError_t launch_transpose_kr(const __nv_bfloat16* mt, __nv_bfloat16* mtk, int K, int r, int num_sms, cudaStream_t s,
                                const float* cvt_src, __nv_bfloat16* cvt_dst, int64_t cvt_rows, float cvt_scale,
                                unsigned* zero, int zero_words) {
  const int64_t work = static_cast<int64_t>(K / 8) * r + cvt_rows * ((r + 7) & ~7);
  int64_t blocks = (work + 255) / 256;
  if (blocks > 8 * static_cast<int64_t>(num_sms)) blocks = 8 * static_cast<int64_t>(num_sms);
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k_transpose_kr, reinterpret_cast<const unsigned short*>(mt),
                                           reinterpret_cast<unsigned short*>(mtk), K, r, cvt_src, cvt_dst, cvt_rows,
                                           cvt_scale, zero, zero_words);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_lora_down(const __nv_bfloat16* in, const __nv_bfloat16* mt, int mt_kmajor, int M, int K, int r,
                             float scale, float* out_f32, __nv_bfloat16* out_bf16, void* ws, int max_ctas,
                             cudaStream_t s, const float* cvt_src, __nv_bfloat16* cvt_dst, int64_t cvt_rows,
                             float cvt_scale, float t_scale) {
  (void)ws;
  const int tiles = (M + 15) / 16;
  const int rp = r <= 16 ? 16 : (r <= 32 ? 32 : (r <= 64 ? 64 : 128));
  int grid = tiles < max_ctas ? tiles : max_ctas;
  if (grid >= 2) grid &= ~1;  // clusters of two: the CTAs sit on whole TPCs, which the pair GEMMs need
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = grid >= 2 ? 2 : 1;
  cudaError_t e = cudaSuccess;
  // mt staged in shared memory when it fits beside the reduction buffer
  const size_t stage_bytes = static_cast<size_t>(rp) * (static_cast<size_t>(K) + 8) * 2;
  // (pays off only when each CTA walks several tiles)
  const bool staged = tiles >= 4 * grid && stage_bytes + 16 * 16 * static_cast<size_t>(rp) * sizeof(float) <= 200 * 1024;
#define QLORA_LD_ST(NT, KM, W, ST)                                                                               \
  do {                                                                                                           \
    const size_t smem = static_cast<size_t>(W) * 16 * rp * sizeof(float) + (ST ? stage_bytes : 0);               \
    e = set_smem_limit_once(k_lora_down<NT, KM, W, ST>, ST ? 227 * 1024 : smem);                                 \
    if (e != cudaSuccess) break;                                                                                 \
    cfg.blockDim = dim3(W * 32);                                                                                 \
    cfg.dynamicSmemBytes = smem;                                                                                 \
    e = cudaLaunchKernelEx(&cfg, k_lora_down<NT, KM, W, ST>, in, mt, M, K, r, scale, out_f32, out_bf16, cvt_src, \
                           cvt_dst, cvt_rows, cvt_scale, t_scale);                                               \
  } while (0)
#define QLORA_LD(NT, KM, W)           \
  do {                                \
    if (staged)                       \
      QLORA_LD_ST(NT, KM, W, true);   \
    else                              \
      QLORA_LD_ST(NT, KM, W, false);  \
  } while (0)
#define QLORA_LD2(NT, W)     \
  do {                       \
    if (mt_kmajor)           \
      QLORA_LD(NT, true, W); \
    else                     \
      QLORA_LD(NT, false, W); \
  } while (0)
  if (rp == 16) QLORA_LD2(2, 16);
  else if (rp == 32) QLORA_LD2(4, 16);
  else if (rp == 64) QLORA_LD2(8, 8);
  else QLORA_LD2(16, 8);
#undef QLORA_LD2
#undef QLORA_LD
#undef QLORA_LD_ST
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

bool lora_down_ks_plan(int M, int K, int r, int num_sms, int* splits, int* chunks_per_split) {
  if (M <= 0 || K <= 0 || r < 1 || r > 16 || num_sms < 1) return false;
  const int rp = r <= 8 ? 8 : 16;
  const int row_blocks = (M + kLdkRows - 1) / kLdkRows;
  if (row_blocks > num_sms) return false;  // more than a wave of row blocks: the persistent kernel
  const int nc = (K + 31) / 32;
  int S = num_sms / row_blocks;
  S = S < 1 ? 1 : (S > kLdkMaxSplits ? kLdkMaxSplits : S);
  int c = (nc + S - 1) / S;
  // the staged slice of mt must fit: more shares when k is long
  while (static_cast<size_t>(rp) * ldk_pitch(c) * 2 > kLdkMaxSliceBytes) {
    if (++S > kLdkMaxSplits) return false;
    c = (nc + S - 1) / S;
  }
  S = (nc + c - 1) / c;  // every share non-empty
  *splits = S;
  *chunks_per_split = c;
  return true;
}

cudaError_t launch_lora_down_ks(const __nv_bfloat16* in, const __nv_bfloat16* mt, int mt_kmajor, int M, int K, int r,
                                float scale, float* out_f32, __nv_bfloat16* out_bf16, int num_sms, cudaStream_t s,
                                const float* cvt_src, __nv_bfloat16* cvt_dst, int64_t cvt_rows, float cvt_scale,
                                float t_scale) {
  int S = 0, cps = 0;
  if (!lora_down_ks_plan(M, K, r, num_sms, &S, &cps)) return cudaErrorInvalidValue;
  const int rp = r <= 8 ? 8 : 16;
  const size_t smem = ldk_smem_bytes(rp, cps, S);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(S), static_cast<unsigned>((M + kLdkRows - 1) / kLdkRows));
  cfg.blockDim = dim3(kLdkThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(S);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaSuccess;
#define QLORA_LDK(NT, KM)                                                                                           \
  do {                                                                                                              \
    e = set_smem_limit_once(k_lora_down_ks<NT, KM>, kLdkMaxSliceBytes + 64 * 1024);                                 \
    if (e == cudaSuccess)                                                                                           \
      e = cudaLaunchKernelEx(&cfg, k_lora_down_ks<NT, KM>, in, mt, M, K, r, cps, scale, out_f32, out_bf16, cvt_src, \
                             cvt_dst, cvt_rows, cvt_scale, t_scale);                                                \
  } while (0)
  if (rp == 8) {
    if (mt_kmajor) QLORA_LDK(1, true); else QLORA_LDK(1, false);
  } else {
    if (mt_kmajor) QLORA_LDK(2, true); else QLORA_LDK(2, false);
  }
#undef QLORA_LDK
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// A 256-thread 1-D launch with programmatic stream serialization (the kernel waits with
// griddep_wait before it touches memory the preceding kernels may still use).
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl_1d(void (*kernel)(KArgs...), int64_t grid, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_silu_mul_fwd(const uint16_t* g, const uint16_t* u, uint16_t* h, int64_t n, int num_sms,
                                cudaStream_t s) {
  const int64_t n2 = n / 2;
  int64_t grid = (n2 + 255) / 256;
  if (grid > num_sms * 16) grid = num_sms * 16;
  if (grid < 1) grid = 1;
  const cudaError_t e = launch_pdl_1d(k_silu_mul_fwd, grid, s, reinterpret_cast<const uint32_t*>(g),
                                      reinterpret_cast<const uint32_t*>(u), reinterpret_cast<uint32_t*>(h), n2);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_silu_mul_bwd(const uint16_t* dh, const uint16_t* g, const uint16_t* u, uint16_t* dg, uint16_t* du,
                                int64_t n, int num_sms, cudaStream_t s) {
  const int64_t n2 = n / 2;
  int64_t grid = (n2 + 255) / 256;
  if (grid > num_sms * 16) grid = num_sms * 16;
  if (grid < 1) grid = 1;
  const cudaError_t e = launch_pdl_1d(k_silu_mul_bwd, grid, s, reinterpret_cast<const uint32_t*>(dh),
                                      reinterpret_cast<const uint32_t*>(g), reinterpret_cast<const uint32_t*>(u),
                                      reinterpret_cast<uint32_t*>(dg), reinterpret_cast<uint32_t*>(du), n2);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qlora
