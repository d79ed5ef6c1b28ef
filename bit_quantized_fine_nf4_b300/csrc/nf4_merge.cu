// Low-rank combinations of a frozen weight with its LoRA branch:
//
//   merge / export   out_bf16[n, k] = bf16( deq(W)[n, k] + s * sum_j B[n, j] A[j, k] )
//   dense update     out_f32[n, k]  = W[n, k] (- deq(Q)[n, k]) + c * sum_j B[n, j] A[j, k]
//   dropout dX       dx[m, k] = bf16(dx[m, k] + (keep(m, k) ? c * sum_j sU[m, j] A[j, k] : 0))
//
// Day 25 notes "Fine-tuning and LoRA/QLoRA", section 2.6: after training the
// product B A is added to W0 and the layer is a plain linear again.  P1 tutorial
// "QLoRA: fine-tuning 7B on a 24 GB card", section 3.8, and the glossary "QLoRA",
// section "Trade-offs": a 4-bit base cannot be merged as is -- dequantise it to
// 16 bits first, merge, and quantise again for serving.  The dense update
// (W - s B A, W - deq(Q)) is the arithmetic of the LoftQ initialisation of the
// same tutorial, section 3.10.
//
// The arithmetic is fixed so the result is reproducible bit for bit:
//   deq(W)[n, k] = bf16_rn(L[code] * a') exactly as the dequantiser computes it;
//   acc = sum over j = 0, 1, ..., r-1 of B[n, j] * A[j, k] in float32, one fused
//         multiply-add per term (B and A are bf16, so every product is exact and
//         each step rounds once, like a separate add);
//   merge:  bf16_rn(deq + s * acc)   (s * acc rounded, then the add rounded);
//   update: (W - deq(Q)) + c * acc   (each operation rounded once in float32).
//
// Layout: a CTA of 8 warps takes a tile of 8 R rows x 256 columns (R = 8, or 4
// for the float32 dense base); warp w owns rows R w .. R w + R - 1, lane l the 8
// columns 8l .. 8l+7 of each.  A[:, tile columns] is staged once in shared
// memory as float32 [r][256], B[tile rows, :] as float32 [r][8 R] (transposed),
// so each term costs two 16-byte loads of A, R/4 broadcast loads of B and 4 R
// packed float32x2 FMAs for 8 R outputs.  The
// weight is HBM traffic (0.516 B per weight read, 2 or 4 B written); the FMA
// chain is r multiply-adds per weight on the CUDA cores.
#include "common.cuh"
#include "kernels.h"

namespace qlora {

constexpr int kMgCols = 256;
constexpr int kMgThreads = 256;

enum MgBase : int { MG_NF4 = 0, MG_F32 = 1, MG_BF16 = 2 };

struct MgParams {
  // NF4 record (the merge base, or the record subtracted by the dense update)
  const uint8_t* codes;
  const int8_t* absq;
  const float* step;
  const float* mean;
  const void* dense;            // dense W [n, k] (float32 or bfloat16), dense update only
  const __nv_bfloat16* lora_a;  // [r, k]
  const __nv_bfloat16* lora_b;  // [n, r] with row stride ldb
  const uint8_t* mask;          // keep bits of [n, k] (masked variant), bit (n k + c) % 8 of byte (n k + c) / 8
  void* out;                    // bf16 (merge, dropout dX) or float32 (update) [n, k]
  int n, k, r, ldb;
  float coef;
};

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// Raw operands of the 8 dequantised weights of one row, columns k .. k+7 (k % 8 == 0): the code
// word, the block's raw scale and its step.
struct Nf4Raw8 {
  uint32_t word;
  int q;
  float step;
};
__device__ __forceinline__ Nf4Raw8 load_raw8(const MgParams& p, int n, int k) {
  const int64_t e0 = static_cast<int64_t>(n) * p.k + k;
  const int64_t b = e0 / 64;
  return {*reinterpret_cast<const uint32_t*>(p.codes + e0 / 2), static_cast<int>(p.absq[b]), p.step[b >> 8]};
}
// The 8 dequantised weights as float32 holding bf16 values: bf16_rn(L[code] * a'), in pairs (one
// packed multiply and one packed round per two weights; each lane rounds like __fmul_rn and
// __float2bfloat16_rn).
__device__ __forceinline__ void deq8(const Nf4Raw8& raw, const float* s_lv, float mu, float (&w)[8]) {
  const float a2 = restore_absmax(static_cast<int8_t>(raw.q), raw.step, mu);
  const float2 aa = make_float2(a2, a2);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // byte i: element 2i in the high nibble, 2i + 1 in the low nibble
    const uint32_t byte = (raw.word >> (8 * i)) & 0xffu;
    const float2 l = make_float2(s_lv[byte >> 4], s_lv[byte & 15u]);
    const float2 v = __fmul2_rn(l, aa);
    const uint32_t pk = pack_bf16x2_rn(v.x, v.y);
    w[2 * i] = __uint_as_float(pk << 16);
    w[2 * i + 1] = __uint_as_float(pk & 0xffff0000u);
  }
}

// ROWS rows x 8 columns per lane; a CTA of 8 warps covers 8 * ROWS rows x 256 columns.
template <int BASE, bool SUB_NF4, bool OUT_BF16, bool MASKED, int ROWS>
__global__ void __launch_bounds__(kMgThreads, 2) k_lowrank_combine(const MgParams p) {
  griddep_wait();  // launched early: dX (in place) and the LoRA matrices may come from the preceding kernels
  griddep_launch_dependents();
  constexpr int kRows = 8 * ROWS;           // rows of the CTA tile
  extern __shared__ float s_mg[];
  float* s_a = s_mg;                        // [r][256]
  float* s_bt = s_a + p.r * kMgCols;        // [r][kRows]
  float* s_lv = s_bt + p.r * kRows;         // [16]
  const int n0 = blockIdx.y * kRows, k0 = blockIdx.x * kMgCols;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kcols = min(kMgCols, p.k - k0);  // a multiple of 64
  // Every HBM read of this thread's ROWS rows x 8 columns is issued first, so its latency
  // overlaps the staging of A and B and the FMA chain (rows past n and lanes past the tile read
  // row n0, column k0 and store nothing).
  const bool lane_on = lane * 8 < kcols;
  const int kc = k0 + (lane_on ? lane * 8 : 0);
  Nf4Raw8 raw[ROWS];
  uint4 dv[ROWS][BASE == MG_F32 ? 2 : 1];
  uint32_t keep8[ROWS];
#pragma unroll
  for (int i = 0; i < ROWS; ++i) {
    const int n = n0 + warp * ROWS + i < p.n ? n0 + warp * ROWS + i : n0;
    const int64_t o = static_cast<int64_t>(n) * p.k + kc;
    if (BASE == MG_NF4 || SUB_NF4) raw[i] = load_raw8(p, n, kc);
    if (BASE == MG_F32) {  // plain loads: the dense input may be the output (in place)
      dv[i][0] = *reinterpret_cast<const uint4*>(static_cast<const float*>(p.dense) + o);
      dv[i][BASE == MG_F32 ? 1 : 0] = *reinterpret_cast<const uint4*>(static_cast<const float*>(p.dense) + o + 4);
    } else if (BASE == MG_BF16) {
      dv[i][0] = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.dense) + o);
    }
    keep8[i] = MASKED ? p.mask[o >> 3] : 0xffu;
  }
  // stage A[:, k0 .. k0 + kcols) and B[n0 .. n0 + kRows, :]^T as float32
  for (int i = threadIdx.x; i < p.r * (kMgCols / 8); i += kMgThreads) {
    const int j = i / (kMgCols / 8), c8 = (i % (kMgCols / 8)) * 8;
    float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
    if (c8 < kcols) {
      const uint4 v = ldg_nc_v4(p.lora_a + static_cast<int64_t>(j) * p.k + k0 + c8);
      lo = make_float4(bf16_bits_to_f32(v.x & 0xffffu), bf16_bits_to_f32(v.x >> 16), bf16_bits_to_f32(v.y & 0xffffu),
                       bf16_bits_to_f32(v.y >> 16));
      hi = make_float4(bf16_bits_to_f32(v.z & 0xffffu), bf16_bits_to_f32(v.z >> 16), bf16_bits_to_f32(v.w & 0xffffu),
                       bf16_bits_to_f32(v.w >> 16));
    }
    *reinterpret_cast<float4*>(s_a + j * kMgCols + c8) = lo;
    *reinterpret_cast<float4*>(s_a + j * kMgCols + c8 + 4) = hi;
  }
  const unsigned short* b16 = reinterpret_cast<const unsigned short*>(p.lora_b);
  for (int i = threadIdx.x; i < p.r * kRows; i += kMgThreads) {
    const int row = i % kRows, j = i / kRows;  // consecutive threads write consecutive banks
    const int n = n0 + row;
    s_bt[j * kRows + row] = n < p.n ? bf16_bits_to_f32(b16[static_cast<int64_t>(n) * p.ldb + j]) : 0.f;
  }
  if (threadIdx.x < 16) {
    constexpr uint32_t hex[16] = QLORA_NF4_LEVELS_HEX;
    uint32_t v = 0;
#pragma unroll
    for (int c = 0; c < 16; ++c) v = threadIdx.x == c ? hex[c] : v;
    s_lv[threadIdx.x] = __uint_as_float(v);
  }
  __syncthreads();

  if (!lane_on) return;
  float2 acc[ROWS][4];
#pragma unroll
  for (int i = 0; i < ROWS; ++i)
#pragma unroll
    for (int h = 0; h < 4; ++h) acc[i][h] = make_float2(0.f, 0.f);
  const float* a_col = s_a + lane * 8;
  const float* b_row = s_bt + warp * ROWS;
  for (int j = 0; j < p.r; ++j) {
    const float4 a0 = *reinterpret_cast<const float4*>(a_col + j * kMgCols);
    const float4 a1 = *reinterpret_cast<const float4*>(a_col + j * kMgCols + 4);
    float bv[ROWS];
#pragma unroll
    for (int i4 = 0; i4 < ROWS; i4 += 4) {
      const float4 bb = *reinterpret_cast<const float4*>(b_row + j * kRows + i4);
      bv[i4] = bb.x;
      bv[i4 + 1] = bb.y;
      bv[i4 + 2] = bb.z;
      bv[i4 + 3] = bb.w;
    }
    const float2 ap[4] = {make_float2(a0.x, a0.y), make_float2(a0.z, a0.w), make_float2(a1.x, a1.y),
                          make_float2(a1.z, a1.w)};
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
      const float2 b2 = make_float2(bv[i], bv[i]);
#pragma unroll
      for (int h = 0; h < 4; ++h) acc[i][h] = __ffma2_rn(b2, ap[h], acc[i][h]);
    }
  }

  const float mu = (BASE == MG_NF4 || SUB_NF4) ? *p.mean : 0.f;
#pragma unroll
  for (int i = 0; i < ROWS; ++i) {
    const int n = n0 + warp * ROWS + i;
    if (n >= p.n) break;
    float base[8];
    if (BASE == MG_NF4) {
      deq8(raw[i], s_lv, mu, base);
    } else {
      if (BASE == MG_F32) {
        const uint32_t wv[8] = {dv[i][0].x, dv[i][0].y, dv[i][0].z, dv[i][0].w,
                                dv[i][BASE == MG_F32 ? 1 : 0].x, dv[i][BASE == MG_F32 ? 1 : 0].y,
                                dv[i][BASE == MG_F32 ? 1 : 0].z, dv[i][BASE == MG_F32 ? 1 : 0].w};
#pragma unroll
        for (int e = 0; e < 8; ++e) base[e] = __uint_as_float(wv[e]);
      } else {
        const uint32_t wv[4] = {dv[i][0].x, dv[i][0].y, dv[i][0].z, dv[i][0].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          base[2 * h] = bf16_bits_to_f32(wv[h] & 0xffffu);
          base[2 * h + 1] = bf16_bits_to_f32(wv[h] >> 16);
        }
      }
      if (SUB_NF4) {
        float qd[8];
        deq8(raw[i], s_lv, mu, qd);
#pragma unroll
        for (int e = 0; e < 8; ++e) base[e] = __fsub_rn(base[e], qd[e]);
      }
    }
    const int64_t o = static_cast<int64_t>(n) * p.k + kc;
    const uint32_t keep = keep8[i];
    float o8[8];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      // base + coef * acc, each operation rounded once (scalar: a packed multiply followed by a
      // packed add may be contracted into one fused operation)
      const float s0 = __fadd_rn(base[2 * h], __fmul_rn(p.coef, acc[i][h].x));
      const float s1 = __fadd_rn(base[2 * h + 1], __fmul_rn(p.coef, acc[i][h].y));
      const bool k0b = p.r > 0 && ((keep >> (2 * h)) & 1u), k1b = p.r > 0 && ((keep >> (2 * h + 1)) & 1u);
      o8[2 * h] = k0b ? s0 : base[2 * h];
      o8[2 * h + 1] = k1b ? s1 : base[2 * h + 1];
    }
    if (OUT_BF16) {
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + o) =
          make_uint4(pack_bf16x2_rn(o8[0], o8[1]), pack_bf16x2_rn(o8[2], o8[3]), pack_bf16x2_rn(o8[4], o8[5]),
                     pack_bf16x2_rn(o8[6], o8[7]));
    } else {
      float* dst = static_cast<float*>(p.out) + o;
      *reinterpret_cast<float4*>(dst) = make_float4(o8[0], o8[1], o8[2], o8[3]);
      *reinterpret_cast<float4*>(dst + 4) = make_float4(o8[4], o8[5], o8[6], o8[7]);
    }
  }
}

template <int BASE, bool SUB_NF4, bool OUT_BF16, bool MASKED = false>
static cudaError_t run_combine(const MgParams& p, cudaStream_t s) {
  // 8 rows per lane (halves the shared-memory loads of A per FMA); the dense updates (a float32
  // base, or a subtracted record) keep 4: their preloaded operands would not fit the registers
  constexpr int ROWS = (BASE == MG_F32 || SUB_NF4) ? 4 : 8;
  constexpr int kRows = 8 * ROWS;
  auto kern = k_lowrank_combine<BASE, SUB_NF4, OUT_BF16, MASKED, ROWS>;
  const size_t smem = (static_cast<size_t>(p.r) * (kMgCols + kRows) + 16) * sizeof(float);
  cudaError_t e = set_smem_limit_once(kern, (128 * (kMgCols + kRows) + 16) * 4);
  if (e != cudaSuccess) return e;
  const dim3 grid((p.k + kMgCols - 1) / kMgCols, (p.n + kRows - 1) / kRows);
  e = launch_pdl_plain(kern, grid, dim3(kMgThreads), smem, s, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_nf4_merge(const Nf4Dev& w, const __nv_bfloat16* lora_a, const __nv_bfloat16* lora_b, int r,
                             float scale, __nv_bfloat16* out, cudaStream_t s) {
  MgParams p = {};
  p.codes = w.codes;
  p.absq = w.absq;
  p.step = w.step;
  p.mean = w.mean;
  p.lora_a = lora_a;
  p.lora_b = lora_b;
  p.out = out;
  p.n = static_cast<int>(w.n);
  p.k = static_cast<int>(w.k);
  p.r = r;
  p.ldb = r;
  p.coef = scale;
  return run_combine<MG_NF4, false, true>(p, s);
}

cudaError_t launch_lowrank_update(const void* dense, int dense_bf16, const Nf4Dev* sub, const __nv_bfloat16* lora_a,
                                  const __nv_bfloat16* lora_b, int r, float coef, float* out, int64_t n, int64_t k,
                                  cudaStream_t s) {
  MgParams p = {};
  if (sub) {
    p.codes = sub->codes;
    p.absq = sub->absq;
    p.step = sub->step;
    p.mean = sub->mean;
  }
  p.dense = dense;
  p.lora_a = lora_a;
  p.lora_b = lora_b;
  p.out = out;
  p.n = static_cast<int>(n);
  p.k = static_cast<int>(k);
  p.r = r;
  p.ldb = r;
  p.coef = coef;
  if (dense_bf16) return sub ? run_combine<MG_BF16, true, false>(p, s) : run_combine<MG_BF16, false, false>(p, s);
  return sub ? run_combine<MG_F32, true, false>(p, s) : run_combine<MG_F32, false, false>(p, s);
}

cudaError_t launch_dropout_lora_dx(__nv_bfloat16* dx, const __nv_bfloat16* su, const __nv_bfloat16* lora_a,
                                   const uint8_t* mask, int M, int K, int r, float coef, cudaStream_t s) {
  MgParams p = {};
  p.dense = dx;
  p.lora_a = lora_a;
  p.lora_b = su;
  p.mask = mask;
  p.out = dx;
  p.n = M;
  p.k = K;
  p.r = r;
  p.ldb = lora_ld(r);
  p.coef = coef;
  return run_combine<MG_BF16, false, true, true>(p, s);
}

}  // namespace qlora
